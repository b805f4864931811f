"""Build libwb.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each CUDA translation unit is compiled in parallel, then linked into
``whisper_encoder_gb300/_build/libwb.so`` (git-ignored); ``--debug`` builds the
bounds-checked variant into ``_build_debug/libwb_debug.so``.  Usage:
    python -m whisper_encoder_gb300.build [--force] [--verbose-ptxas] [--debug]
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libwb.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libwb_debug.so")
SOURCES = ["api.cu", "kernels.cu", "tc_kernels.cu", "static_scratch.cu", "host_pipeline.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags(ptxas_verbose: bool = False, debug: bool = False):
    f = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]
    if debug:
        f.append("-DWB_DEBUG=1")
    if ptxas_verbose:
        f.append("-Xptxas=-v")
    return f


def _digest(debug: bool = False) -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    with open(os.path.join(ROOT, "include", "wb.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(_flags(debug=debug)).encode())
    return h.hexdigest()


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True, debug: bool = False) -> str:
    """Compile (if sources changed) and return the path of libwb.so.

    debug=True builds the bounds-checked variant (-DWB_DEBUG) as _build_debug/libwb_debug.so."""
    out_dir = BUILD_DEBUG if debug else BUILD
    lib_path = LIB_DEBUG if debug else LIB
    os.makedirs(out_dir, exist_ok=True)
    stamp = os.path.join(out_dir, "digest.txt")
    dg = _digest(debug)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp) and open(stamp).read() == dg:
        return lib_path
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *_flags(ptxas_verbose, debug), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for obj, log in ex.map(compile_one, SOURCES):
            objs.append(obj)
            if log and (ptxas_verbose or not quiet):
                sys.stderr.write(log)
    tmp = lib_path + ".tmp"
    cmd = [nvcc, ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as fh:
        fh.write(dg)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_verbose="--verbose-ptxas" in sys.argv, quiet=False,
                debug="--debug" in sys.argv))
