"""CPU checks of the C ABI: libwb builds for sm_103a, loads, exports every
function include/wb.h declares, and rejects bad arguments on the host before
touching the GPU.  Also checks that the product path and the oracle share no
code.  No compute call is made here (no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from whisper_encoder_gb300 import build
    build.build()
    from whisper_encoder_gb300 import _lib
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "wb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(wb_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported_and_bound(lib):
    from whisper_encoder_gb300 import _lib
    names = declared_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"
    assert set(_lib.SIGNATURES) == set(names)


def test_header_constants_match_binding():
    from whisper_encoder_gb300 import _lib
    src = open(os.path.join(ROOT, "include", "wb.h")).read()
    consts = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"#define\s+(WB_[A-Z0-9_]+)\s+(0x[0-9A-Fa-f]+|\d+)u?\b", src)}
    assert consts["WB_SELFTEST_WAIT_SITE"] == _lib.WB_SELFTEST_WAIT_SITE
    assert consts["WB_SELFTEST_BOUNDS_SITE"] == _lib.WB_SELFTEST_BOUNDS_SITE
    assert consts["WB_LOGMEL_STATIC_MAX_CHUNKS"] == _lib.WB_LOGMEL_STATIC_MAX_CHUNKS
    assert 0 < _lib.WB_SELFTEST_WAIT_SITE < 256   # bits 8..15 of the error word


def test_status_strings_and_version(lib):
    from whisper_encoder_gb300 import _lib
    assert lib.wb_version() >= 100
    for code, word in [(0, "ok"), (-1, "invalid"), (-4, "timed out"), (-5, "workspace"), (-6, "bounds")]:
        assert word in _lib.status_string(code)


def test_workspace_queries_are_host_only(lib):
    from whisper_encoder_gb300 import _lib
    import synthetic
    d = synthetic.LARGE_V3
    dims = _lib.wb_dims(d.n_mels, d.d_model, d.n_heads, d.n_layers, d.d_ffn)
    bf = _lib.wb_precision(0, 0, 0, 0, 0, 0)
    f8 = _lib.wb_precision(1, 1, 0, 0, 1, 1)
    w_bf = lib.wb_encoder_workspace_bytes(ctypes.byref(dims), 32, ctypes.byref(bf))
    w_f8 = lib.wb_encoder_workspace_bytes(ctypes.byref(dims), 32, ctypes.byref(f8))
    M = 32 * 1500
    assert w_bf >= M * 1280 * 2 * 6 + M * 5120 * 2
    assert w_f8 >= w_bf + M * 5120          # E4M3 copies of the activations
    assert lib.wb_logmel_workspace_bytes(32, 128) > 32 * 3 * 480400 * 2
    assert lib.wb_logmel_workspace_bytes(0, 128) == 0
    assert lib.wb_conv_stem_workspace_bytes(ctypes.byref(dims), 32) >= 32 * 3001 * 1280 * 2
    bad = _lib.wb_dims(128, 1000, 20, 32, 5120)                       # d != 64 * heads
    assert lib.wb_encoder_workspace_bytes(ctypes.byref(bad), 32, ctypes.byref(bf)) == 0


def test_argument_errors_return_before_any_launch(lib):
    from whisper_encoder_gb300 import _lib
    import synthetic
    d = synthetic.TINY
    dims = _lib.wb_dims(d.n_mels, d.d_model, d.n_heads, d.n_layers, d.d_ffn)
    fake = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced on these paths
    # log-mel: bad mel count, negative sizes, too-small workspace
    assert lib.wb_logmel(fake, 480000, 480000, 1, 7, fake, fake, 1 << 30, None) == _lib.WB_EINVAL
    assert lib.wb_logmel(fake, -1, 480000, 1, 80, fake, fake, 1 << 30, None) == _lib.WB_EINVAL
    assert lib.wb_logmel(fake, 480000, 480000, 1, 80, fake, fake, 16, None) == _lib.WB_EWORKSPACE
    assert lib.wb_logmel(None, 480000, 480000, 0, 80, None, None, 0, None) == _lib.WB_OK   # empty batch
    # encoder: mixed bf16 x E4M3 site, bad layer range, aliasing output, bad dims
    mixed = _lib.wb_precision(1, 0, 0, 0, 0, 0)
    assert lib.wb_encoder_forward(fake, 1, ctypes.byref(dims), None, None, ctypes.byref(mixed), 0, 1, 0, fake, fake,
                                  1 << 30, None) == _lib.WB_EUNSUPPORTED
    bf = _lib.wb_precision(0, 0, 0, 0, 0, 0)
    assert lib.wb_encoder_forward(fake, 1, ctypes.byref(dims), None, None, ctypes.byref(bf), 0, 2, 0, fake, fake,
                                  1 << 30, None) == _lib.WB_EINVAL
    assert lib.wb_encoder_forward(fake, 1, ctypes.byref(dims), None, None, ctypes.byref(bf), 0, 0, 0, fake, fake,
                                  1 << 30, None) == _lib.WB_EINVAL
    bad = _lib.wb_dims(80, 384, 5, 1, 1536)
    assert lib.wb_encoder_forward(fake, 1, ctypes.byref(bad), None, None, ctypes.byref(bf), 0, 1, 0, fake, fake,
                                  1 << 30, None) == _lib.WB_EINVAL
    # linear: N not a multiple of 32, unknown dtype, misaligned pointer, E4M3 without scales
    assert lib.wb_linear(fake, fake, 16, 33, 64, 0, None, None, None, 0, None, fake, None) == _lib.WB_EINVAL
    assert lib.wb_linear(fake, fake, 16, 32, 64, 7, None, None, None, 0, None, fake, None) == _lib.WB_EUNSUPPORTED
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert lib.wb_linear(odd, fake, 16, 32, 64, 0, None, None, None, 0, None, fake, None) == _lib.WB_EINVAL
    assert lib.wb_linear(fake, fake, 16, 32, 64, 1, None, None, None, 0, None, fake, None) == _lib.WB_EINVAL
    # layernorm: width not a multiple of 128; attention: T beyond the padded V^T rows
    assert lib.wb_layernorm(fake, None, fake, fake, 4, 200, 1e-5, fake, None, None) == _lib.WB_EINVAL
    assert lib.wb_attention(fake, fake, fake, 1, 1505, 2, fake, fake, 1 << 30, None) == _lib.WB_EINVAL
    assert lib.wb_quantize_fp8(fake, -1, fake, fake, None) == _lib.WB_EINVAL
    # LayerNorm fold: width not a multiple of 8, missing gamma, misaligned output, nothing to do
    assert lib.wb_fold_layernorm(fake, None, fake, fake, 16, 12, fake, fake, fake, None) == _lib.WB_EINVAL
    assert lib.wb_fold_layernorm(fake, None, None, fake, 16, 64, fake, fake, fake, None) == _lib.WB_EINVAL
    assert lib.wb_fold_layernorm(fake, None, fake, fake, 16, 64, odd, fake, fake, None) == _lib.WB_EINVAL
    assert lib.wb_fold_layernorm(None, None, None, None, 0, 64, None, None, None, None) == _lib.WB_OK
    # LayerNorm to E4M3: no item size, bad width, missing statistics, misaligned codes, no rows
    assert lib.wb_layernorm_e4m3(fake, fake, fake, 4, 256, 1e-5, 0, fake, fake, fake, None) == _lib.WB_EINVAL
    assert lib.wb_layernorm_e4m3(fake, fake, fake, 4, 200, 1e-5, 4, fake, fake, fake, None) == _lib.WB_EINVAL
    assert lib.wb_layernorm_e4m3(fake, fake, fake, 4, 256, 1e-5, 4, fake, fake, None, None) == _lib.WB_EINVAL
    assert lib.wb_layernorm_e4m3(fake, fake, fake, 4, 256, 1e-5, 4, odd, fake, fake, None) == _lib.WB_EINVAL
    assert lib.wb_layernorm_e4m3(None, None, None, 0, 256, 1e-5, 1, None, None, None, None) == _lib.WB_OK


def test_encode_host_argument_errors(lib):
    # host-side checks of wb_encode_host, all before any copy or launch is queued
    from whisper_encoder_gb300 import _lib
    import synthetic
    d = synthetic.TINY
    hp = _lib.wb_host_pipeline()
    hp.dims = _lib.wb_dims(d.n_mels, d.d_model, d.n_heads, d.n_layers, d.d_ffn)
    hp.batch, hp.samples_per_batch, hp.chunk_stride = 1, 480000, 480000
    fake = 1 << 20
    stem, ln = _lib.wb_stem_weights(fake, fake, fake, fake), _lib.wb_ln_weights(fake, fake)
    layers = (_lib.wb_layer_weights * 1)()
    hp.stem, hp.layers, hp.ln_post = ctypes.pointer(stem), layers, ctypes.pointer(ln)
    hp.dev_audio[0] = hp.dev_audio[1] = hp.dev_out[0] = hp.dev_out[1] = fake
    hp.dev_mel = hp.dev_x0 = fake
    arr = (ctypes.c_void_p * 1)(fake)
    enc = lib.wb_encode_host
    assert enc(ctypes.byref(hp), arr, arr, 0, None) == _lib.WB_OK                 # nothing to do
    assert enc(None, arr, arr, 1, None) == _lib.WB_EINVAL
    assert enc(ctypes.byref(hp), arr, arr, -1, None) == _lib.WB_EINVAL
    assert enc(ctypes.byref(hp), None, arr, 1, None) == _lib.WB_EINVAL            # no host audio
    nulls = (ctypes.c_void_p * 1)(None)
    assert enc(ctypes.byref(hp), arr, nulls, 1, None) == _lib.WB_EINVAL           # a missing host output
    hp.upload_stream = fake                                                       # only one copy stream
    assert enc(ctypes.byref(hp), arr, arr, 1, None) == _lib.WB_EINVAL
    hp.download_stream = fake
    hp.dev_out[1] = None                                                          # second buffer missing
    assert enc(ctypes.byref(hp), arr, arr, 1, None) == _lib.WB_EINVAL
    hp.batch = 0
    assert enc(ctypes.byref(hp), arr, arr, 1, None) == _lib.WB_EINVAL


def _imports(path):
    out = []
    for dirpath, _, files in os.walk(path):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                out += re.findall(r"^\s*(?:from|import)\s+([\w\.]+)", src, flags=re.M)
                out += re.findall(r'#include\s+"([^"]+)"', src)
    return out


def test_product_and_oracle_share_no_code():
    prod = _imports(os.path.join(ROOT, "whisper_encoder_gb300"))
    assert not [m for m in prod if m.startswith("oracle") or "oracle" in m], prod
    orc = _imports(os.path.join(ROOT, "oracle"))
    assert not [m for m in orc if "whisper_encoder_gb300" in m or m.startswith("synthetic")], orc
    # the shared input module holds no step of the method (no FFT, mel, norm or softmax code)
    src = open(os.path.join(ROOT, "synthetic", "__init__.py")).read()
    for word in ("fft", "mel_", "log10", "softmax", "layer_norm", "erf"):
        assert word not in src, word


def test_header_is_plain_c(tmp_path):
    # include/wb.h must serve C callers: it compiles as C99 on its own (no CUDA headers, no C++), and
    # every function it declares has a prototype a C translation unit can take the address of
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "use_wb.c"
    src.write_text('#include "wb.h"\n#include <stdio.h>\nint main(void) {\n  void* fns[] = {\n'
                   + "".join(f"    (void*){n},\n" for n in names)
                   + '  };\n  printf("%d\\n", (int)(sizeof(fns) / sizeof(fns[0])));\n  return 0;\n}\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-Wno-pedantic",
                        "-I" + os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "use_wb.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
