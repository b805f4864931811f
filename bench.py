#!/usr/bin/env python3
"""Throughput of the Whisper large-v3 encoder hot path on GB300.

One step = wb_logmel + wb_conv_stem + wb_encoder_forward (32 layers + final
LayerNorm) over one batch of 32 seeded synthetic 30 s chunks whose audio is
already resident in device memory.  Metric: audio-seconds processed per
second (RTFx).  Under torchrun every rank runs an independent replica on its
own 32 chunks (no data-path collective; weak scaling); the host-side barrier
and a MAX all-reduce of the elapsed time are the only cross-rank traffic.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--precision bf16|mixed_fp8|aggressive_fp8]
                    [--batch B] [--impl wb|reference]

--impl reference times the float64 CPU oracle (the reference arm of this
build) on the host cores, one chunk through log-mel, stem and one encoder
layer per step, extrapolated to the 32-layer model.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "encoder audio-sec/s (RTFx) at large-v3 batch 32; % of tensor-core peak"
UNIT = "audio-s/s"
CHUNK_S = 30.0


def flops_per_chunk(dims) -> dict:
    """Algorithmic FLOPs of one 30 s chunk by kernel class (multiply-add = 2)."""
    T, d, F, C, H = 1500, dims.d_model, dims.d_ffn, dims.n_mels, dims.n_heads
    L = dims.n_layers
    return {
        "logmel.dft": 2.0 * 3000 * 402 * 400,
        "logmel.mel": 2.0 * 3000 * C * 201,
        "stem.conv1": 2.0 * 3000 * d * 3 * C,
        "stem.conv2": 2.0 * 1500 * d * 3 * d,
        "enc.qkv": L * 2.0 * T * d * 3 * d,
        "enc.attention": L * 4.0 * H * T * T * 64,
        "enc.out_proj": L * 2.0 * T * d * d,
        "enc.fc1": L * 2.0 * T * d * F,
        "enc.fc2": L * 2.0 * T * F * d,
    }


def bytes_per_chunk(dims, precision: str = "bf16") -> dict:
    """Algorithmic HBM bytes of the bandwidth-bound classes per chunk (bf16 activations)."""
    T, d, F, C = 1500, dims.d_model, dims.d_ffn, dims.n_mels
    L = dims.n_layers
    row = T * d * 2.0                                   # one [1500, d] bf16 tensor
    out = {"logmel.post": 2.0 * C * 3000 * 4,           # clamp + scale in place
           "logmel.prep": 480000 * 4 + 3 * 480400 * 2.0}   # audio in, padded split-bf16 copy out
    if precision == "bf16":
        # LN1 / LN2 folded into QKV / FC1: the statistics kernels read each row once; the final LN reads + writes
        out["enc.layernorm"] = 2 * L * row + 2 * row
    else:
        # LN1 / LN2 write E4M3 codes straight from the bf16 rows (read [1500, d] bf16, write u8);
        # the final LN reads and writes bf16
        out["enc.layernorm"] = 2 * L * (row + row / 2) + 2 * row
        # E4M3 copy of the FC2 input ([1500, F]): read bf16, write u8
        out["enc.quantize"] = L * (T * F * 2.0 + T * F)
        if precision == "aggressive_fp8":   # and of the out-projection input (read bf16, write u8)
            out["enc.quantize"] += L * (row + row / 2)
    return out


def step_roofline(fl: dict, by: dict, B: int, peaks: dict, fp8_classes: set, ms_step: float) -> dict:
    """Roofline time of one step: sum over kernel classes of max(FLOPs / peak, bytes / HBM bandwidth)."""
    t = 0.0
    for c in set(fl) | set(by):
        tf = fl.get(c, 0.0) * B / (peaks["bf16_sustained"] * 1e12 * (2.0 if c in fp8_classes else 1.0))
        tb = by.get(c, 0.0) * B / (peaks["hbm_gbs"] * 1e9)
        t += max(tf, tb)
    return {"ideal_ms": round(t * 1e3, 3), "frac": round(t * 1e3 / ms_step, 4),
            "peaks": f"{peaks['source']}: bf16 sustained {peaks['bf16_sustained']} TFLOP/s (x2 for E4M3 GEMM "
                     f"classes), HBM {peaks['hbm_gbs']} GB/s"}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from an ncu capture of the
# kernel class at the batch-32 shape (profiles/); None where the code changed since the capture.
TRAFFIC = {"enc.attention": 473.3e6}


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                               parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.f.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_uuid(torch, dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ----------------------------------------------------------------------------- CPU oracle
def oracle_chunk_seconds(dims, seed: int, n_layers_sample: int = 1) -> tuple[float, dict]:
    """Time the float64 oracle on one chunk: log-mel, stem, n sample layers, one LN.

    Returns the extrapolated seconds per chunk for the full model and the parts.
    """
    from oracle import encoder as oenc
    from oracle import frontend as ofe
    w = synthetic.encoder_weights(dims, seed, "bf16", n_layers=n_layers_sample)
    x = synthetic.tone_chunk(seed)
    t0 = time.perf_counter()
    mel = ofe.log_mel(x, dims.n_mels)
    t1 = time.perf_counter()
    h = oenc.conv_stem(mel, w)
    t2 = time.perf_counter()
    for L in w["layers"]:
        h = oenc.encoder_layer(h, L, dims.n_heads)
    t3 = time.perf_counter()
    oenc.layer_norm(h, w["layers"][0]["ln1_g"], w["layers"][0]["ln1_b"])
    t4 = time.perf_counter()
    per_layer = (t3 - t2) / n_layers_sample
    total = (t1 - t0) + (t2 - t1) + dims.n_layers * per_layer + (t4 - t3)
    return total, {"logmel_s": t1 - t0, "stem_s": t2 - t1, "layer_s": per_layer, "final_ln_s": t4 - t3}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_info() -> dict:
    """Host threads the oracle may use: all cores, the affinity mask, the BLAS thread setting."""
    blas = {k: os.environ[k] for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS") if k in os.environ}
    return {"os_cpu_count": os.cpu_count(), "affinity_cpus": cpu_cores(),
            "blas_threads": blas or "library default (all cores)"}


def run_reference(args) -> None:
    """The reference arm: the float64 oracle on the host cores.

    A step is one of the 32 encoder layers of one 30 s chunk (1/32 of the chunk's encoder work, the
    oracle's dominant cost); the chunk's front end (log-mel, conv stem) and final LayerNorm are timed
    once beforehand.  value = 30 s / (front end + 32 x median layer time), so value x ms_per_step is
    about 30/32 audio-seconds per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import encoder as oenc
    from oracle import frontend as ofe
    dims = synthetic.LARGE_V3
    seed = synthetic.SEED_LARGE_B32
    w = synthetic.encoder_weights(dims, seed, "bf16", n_layers=1)
    x = synthetic.tone_chunk(seed)
    t0 = time.perf_counter()
    x0 = oenc.conv_stem(ofe.log_mel(x, dims.n_mels), w)
    oenc.layer_norm(x0, w["layers"][0]["ln1_g"], w["layers"][0]["ln1_b"])
    t_front = time.perf_counter() - t0
    per_step = []
    h = x0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        h = oenc.encoder_layer(h, w["layers"][0], dims.n_heads)
        t = time.perf_counter() - t0
        if i >= args.warmup:
            per_step.append(t)
    t_layer = statistics.median(per_step)
    value = CHUNK_S / (t_front + dims.n_layers * t_layer)
    sample = ("per step: one of the 32 encoder layers of one 30 s chunk (large-v3 shapes) through the float64 "
              f"oracle, {t_layer:.3f} s; the chunk's log-mel, conv stem and final LayerNorm timed once "
              f"({t_front:.3f} s); value = 30 s / (front end + 32 x layer)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_layer * 1000.0, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(args, 1),
        "step_unit": "one of the 32 encoder layers of one 30 s chunk (30/32 audio-seconds of encoder work)",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample,
                         "host": cpu_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def replica_seed(base: int, rank: int, batch: int) -> int:
    """Rank r of an N-replica run encodes its own chunks base + r*batch ... base + r*batch + batch - 1."""
    return base + rank * batch


def job_throughput(local_ms: float, steps: int, batch: int, world: int, reduce_max) -> tuple[float, float]:
    """Whole-job audio-s/s: every rank's chunks over the slowest rank's time.

    ``reduce_max`` maps this rank's elapsed milliseconds to the maximum over
    ranks (identity on one process).  Returns (value, ms per step)."""
    ms_step = reduce_max(local_ms) / steps
    return world * batch * CHUNK_S / (ms_step / 1000.0), ms_step


def workload_name(args) -> str:
    return (f"whisper large-v3 encoder hot path: log-mel + conv stem + 32 layers + final LN, "
            f"batch {args.batch} x 30 s synthetic chunks, {args.precision}")


def arm_config(args, world: int) -> dict:
    return {"workload": workload_name(args), "global_batch": world * args.batch, "seq_len": 1500,
            "parallelism": f"replicas x{world}", "l2": "flushed (256 MB write) between timed steps"}


def run_case(args) -> None:
    """Launch one kernel class at its batch-32 large-v3 shape three times (for ncu captures) and time it."""
    import torch
    import whisper_encoder_gb300 as wb
    wb.load()
    dims, B = synthetic.LARGE_V3, args.batch
    M, d, F, H = B * 1500, dims.d_model, dims.d_ffn, dims.n_heads
    g = torch.Generator(device="cuda").manual_seed(0)

    def rnd(*shape, scale=1.0):
        return (torch.randn(*shape, device="cuda", generator=g) * scale).to(torch.bfloat16)

    if args.case in ("fc1", "fc2", "qkv", "out", "fc1_e4m3", "fc2_e4m3", "qkv_e4m3"):
        base = args.case.replace("_e4m3", "")
        n, k = {"fc1": (F, d), "fc2": (d, F), "qkv": (3 * d, d), "out": (d, d)}[base]
        a, w = rnd(M, k), rnd(n, k, scale=0.02)
        bias = torch.zeros(n, device="cuda")
        resid = rnd(M, n) if base in ("out", "fc2") else None           # the encoder's residual epilogue
        if args.case.endswith("_e4m3"):
            # E4M3 operands with per-tensor scales (the mixed_fp8 qkv / ffn sites)
            (qa, sa), (qw, sw) = wb.quantize_fp8(a), wb.quantize_fp8(w)
            fn = lambda: wb.linear(qa, qw, bias=bias, scale_a=sa, scale_w=sw, gelu=base == "fc1",  # noqa: E731
                                   resid=resid)
        else:
            fn = lambda: wb.linear(a, w, bias=bias, gelu=base == "fc1", resid=resid)  # noqa: E731
        flops = 2.0 * M * n * k
    elif args.case == "attention":
        q, k_, v = rnd(B, 1500, d), rnd(B, 1500, d), rnd(B, 1500, d)
        fn = lambda: wb.attention(q, k_, v, H)  # noqa: E731
        flops = 4.0 * B * H * 1500 * 1500 * 64
    elif args.case == "layernorm":
        x = rnd(M, d)
        gam = torch.ones(d, device="cuda")
        bet = torch.zeros(d, device="cuda")
        fn = lambda: wb.layernorm(x, gam, bet)  # noqa: E731
        flops = 2.0 * M * d * 2      # bytes moved (read + write), reported in the same field
    elif args.case == "layernorm_e4m3":
        # LayerNorm straight to E4M3 codes with one scale per 1500-row chunk (the mixed_fp8 LN1 / LN2 sites)
        x = rnd(M, d, scale=2.0)
        gam = torch.ones(d, device="cuda")
        bet = torch.zeros(d, device="cuda")
        fn = lambda: wb.layernorm_e4m3(x, gam, bet, rows_per_item=1500)  # noqa: E731
        flops = M * d * 2.0 + M * d      # bytes: bf16 rows read, E4M3 codes written
    elif args.case == "longform":
        # 45 min of synthetic audio in 30 s windows at a 25 s stride (the PyPI page's overlapping-chunk
        # mode): 108 windows through the same three calls in 3 batches of 36, audio already on the device
        stride, per = 400000, 36
        x = synthetic.long_audio(synthetic.SEED_LONGFORM)
        n = 1 + max(0, -(-(len(x) - 480000) // stride))
        stem, enc = wb.upload_weights(synthetic.encoder_weights(dims, synthetic.SEED_LONGFORM, "bf16"))
        xd = torch.from_numpy(x).cuda()
        pipe = wb.Pipeline(dims, stem, enc, batch=per)

        def fn():
            for i in range(0, n, per):
                pipe(xd[i * stride:], chunk_stride=stride, n_chunks=min(per, n - i))
        fn()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(3):
            fn()
        ev[1].record()
        torch.cuda.synchronize()
        ms = ev[0].elapsed_time(ev[1]) / 3
        audio_s = len(x) / 16000.0
        print(json.dumps({"case": "longform", "windows": n, "audio_s": audio_s, "ms": round(ms, 3),
                          "audio_s_per_s": round(audio_s / (ms / 1000.0), 1)}))
        return
    elif args.case == "logmel":
        audio = torch.randn(B * 480000, device="cuda", generator=g) * 0.1
        fn = lambda: wb.logmel(audio, B, dims.n_mels)  # noqa: E731
        flops = B * (2.0 * 3000 * 402 * 400 + 2.0 * 3000 * dims.n_mels * 201)
    else:
        raise SystemExit(f"unknown case {args.case}")
    fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(3):
        fn()
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / 3
    rate = flops / (ms / 1000)
    hbm = args.case.startswith("layernorm")
    print(json.dumps({"case": args.case, "batch": B, "ms": round(ms, 4),
                      ("gbs" if hbm else "tflops"): round(rate / (1e9 if hbm else 1e12), 1)}))


# ----------------------------------------------------------------------------- GPU arm
def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--precision", choices=("bf16", "mixed_fp8", "aggressive_fp8"), default="bf16")
    ap.add_argument("--impl", choices=("wb", "reference"), default="wb")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mixed-fp8", action="store_true",
                    help="skip the mixed_fp8 step timed after the bf16 one (bf16 runs only)")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the batch-1 CUDA-graph and 45-minute long-form workloads timed after the bf16 step")
    ap.add_argument("--graph", action="store_true", help="replay each step from a CUDA graph of the three calls")
    ap.add_argument("--case", choices=("fc1", "fc2", "qkv", "out", "fc1_e4m3", "fc2_e4m3", "qkv_e4m3", "attention",
                                       "layernorm", "layernorm_e4m3", "logmel", "longform"),
                    default=None,
                    help="launch one kernel class at full size (for profiler captures) instead of the bench")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from whisper_encoder_gb300 import build as wbuild
    if rank == 0 or world == 1:
        wbuild.build()
    if dist is not None:
        dist.barrier()
    import whisper_encoder_gb300 as wb

    dims = synthetic.LARGE_V3
    B = args.batch
    precision = {"bf16": wb.PRESET_BF16, "mixed_fp8": wb.PRESET_MIXED_FP8,
                 "aggressive_fp8": wb.PRESET_AGGRESSIVE_FP8}[args.precision]
    seed = synthetic.SEED_LARGE_B32
    host_w = synthetic.encoder_weights(dims, seed, "bf16")
    stem, enc = wb.upload_weights(host_w)
    del host_w
    audio_np = synthetic.tone_batch(replica_seed(seed, rank, B), B).reshape(-1)
    audio = torch.from_numpy(audio_np).cuda()
    pipe = wb.Pipeline(dims, stem, enc, B, precision)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")   # > 129 MB L2
    peaks = load_peaks()
    fl = flops_per_chunk(dims)

    def reduce_max(v: float) -> float:
        t = torch.tensor([v], dtype=torch.float64, device="cuda")
        if dist is not None:
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return t.item()

    def timed(pipe_, graph_mode: bool) -> dict:
        """Warm up, then time K steps (L2 flushed before each) with CUDA events on the launching
        stream, the library's per-launch events and the clock sampler running."""
        step = (lambda: pipe_(audio))  # noqa: E731
        graph_launches = None
        if graph_mode:
            wb.profile_begin()                       # count the library's launches in one eager step
            pipe_(audio)
            torch.cuda.synchronize()
            graph_launches = sum(n for _, n in wb.profile_end().values())
            graph = pipe_.capture(audio)
            step = graph.replay
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if wb.check_device_error() != 0:
            raise RuntimeError("device error during warm-up")
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        sampler = ClockSampler(gpu_uuid(torch, local))
        time.sleep(0.3)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        if not graph_mode:
            wb.profile_begin()
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            stops[k].record(stream)
        torch.cuda.synchronize()
        prof = wb.profile_end() if not graph_mode else {}
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop()
        total_ms = sum(s_.elapsed_time(e_) for s_, e_ in zip(starts, stops))
        if wb.check_device_error() != 0:
            raise RuntimeError("device error in the timed region")
        value, ms_step = job_throughput(total_ms, args.steps, B, world, reduce_max)
        launches = sum(n for _, n in prof.values()) if prof else graph_launches * args.steps
        return {"value": value, "ms_step": ms_step, "total_ms": total_ms, "prof": prof, "clocks": clocks,
                "gpu_launches": launches}

    def analyse(res: dict, prec: str) -> dict:
        """Per-class rates, the dominant tensor-core class against its peak, and the step roofline."""
        prof, total_ms = res["prof"], res["total_ms"]
        fp8_classes = {"mixed_fp8": {"enc.qkv", "enc.fc1", "enc.fc2"},
                       "aggressive_fp8": {"enc.qkv", "enc.out_proj", "enc.fc1", "enc.fc2"}}.get(prec, set())
        kernels = {}
        for name, (ms, n) in prof.items():
            per_step_ms = ms / args.steps
            kernels[name] = {"ms_per_step": round(per_step_ms, 4), "launches_per_step": n // args.steps,
                             "share": round(ms / max(total_ms, 1e-9), 4)}
            if name in fl:
                tf = fl[name] * B / (per_step_ms / 1000.0) / 1e12
                pk = peaks["bf16_sustained"] * (2.0 if name in fp8_classes else 1.0)
                kernels[name]["tflops"] = round(tf, 1)
                kernels[name]["frac"] = round(tf / pk, 4)
                kernels[name]["operands"] = "e4m3" if name in fp8_classes else "bf16"
        roofline = None
        tensor_classes = [c for c in prof if c in fl]
        if tensor_classes:
            dom = max(tensor_classes, key=lambda c: prof[c][0])
            dom_ms, dom_n = prof[dom]
            per_launch_ms = dom_ms / dom_n
            flops_launch = fl[dom] * B / (dom_n / args.steps)
            achieved = flops_launch / (per_launch_ms / 1000.0) / 1e12
            peak = peaks["bf16_sustained"] * (2.0 if dom in fp8_classes else 1.0)
            roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                        "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": TRAFFIC.get(dom),
                        "flops_per_launch": flops_launch, "ms_per_launch": round(per_launch_ms, 4),
                        "peak_source": f"{peaks['source']} bf16 sustained"
                                       + (" x2 (E4M3 nominal ratio)" if dom in fp8_classes else "")}
        step_roof = step_roofline(fl, bytes_per_chunk(dims, prec), B, peaks, fp8_classes, res["ms_step"])
        return {"kernels": kernels, "roofline": roofline, "step_roofline": step_roof}

    res = timed(pipe, args.graph)
    value, ms_step = res["value"], res["ms_step"]

    # ---- end to end: pinned host audio in, encoder output back to pinned host memory, every step.
    # Eager: Pipeline.run_host overlaps each step's upload and download with its neighbours' compute
    # (two device buffers each, copy streams).  Graph: the captured buffers, copies in line.
    audio_host = torch.from_numpy(audio_np).pin_memory()
    out_host = torch.empty(pipe.out.shape, dtype=pipe.out.dtype).pin_memory()
    graph_e2e = pipe.capture(audio) if args.graph else None

    def e2e_steps(k):
        if args.graph:
            for _ in range(k):
                audio.copy_(audio_host, non_blocking=True)
                graph_e2e.replay()
                out_host.copy_(pipe.out, non_blocking=True)
        else:
            pipe.run_host([audio_host] * k, [out_host] * k)

    e2e_steps(2)
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    e_start.record(stream)
    e2e_steps(args.steps)
    e_stop.record(stream)
    torch.cuda.synchronize()
    e2e_value, _ = job_throughput(e_start.elapsed_time(e_stop), args.steps, B, world, reduce_max)
    e2e = {"value": round(e2e_value, 2), "unit": UNIT,
           "h2d_bytes_per_step": audio_host.numel() * audio_host.element_size(),
           "d2h_bytes_per_step": out_host.numel() * out_host.element_size()}

    an = analyse(res, args.precision)
    step_flops = sum(fl.values()) * B
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if args.precision == "bf16" else "bf16+e4m3", "data": "synthetic",
        "impl": "wb",
        "config": arm_config(args, world),
        "tflops": round(step_flops / (ms_step / 1000.0) / 1e12, 1),
        "roofline": an["roofline"], "step_roofline": an["step_roofline"], "e2e": e2e,
        "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "graph": bool(args.graph),
        "kernels": an["kernels"],
    }

    # ---- the same step with the mixed_fp8 preset (E4M3 operands at the qkv and ffn sites, one
    # scale per chunk), same inputs, same number of steps, L2 flush and clock sampling
    if args.precision == "bf16" and not args.graph and not args.no_mixed_fp8:
        del pipe
        torch.cuda.empty_cache()
        pipe8 = wb.Pipeline(dims, stem, enc, B, wb.PRESET_MIXED_FP8)
        res8 = timed(pipe8, False)
        an8 = analyse(res8, "mixed_fp8")
        gemm_fracs = {c: an8["kernels"][c]["frac"] for c in ("enc.qkv", "enc.out_proj", "enc.fc1", "enc.fc2")
                      if c in an8["kernels"]}
        line["mixed_fp8"] = {
            "workload": workload_name(argparse.Namespace(batch=B, precision="mixed_fp8")),
            "value": round(res8["value"], 2), "unit": UNIT, "ms_per_step": round(res8["ms_step"], 3),
            "dtype": "bf16+e4m3", "tflops": round(step_flops / (res8["ms_step"] / 1000.0) / 1e12, 1),
            "gemm_fracs": gemm_fracs,
            "gemm_peaks": "E4M3 classes (qkv, fc1, fc2) against 2 x the measured sustained bf16 peak; "
                          "out_proj (bf16 in mixed_fp8) against 1 x",
            "roofline": an8["roofline"], "step_roofline": an8["step_roofline"],
            "gpu_launches": res8["gpu_launches"], "clocks": res8["clocks"], "kernels": an8["kernels"]}
        del pipe8

    # ---- the other two workloads of the encoder hot path, timed the same way: one chunk at a time
    # replayed from a CUDA graph, and 45 minutes of audio in 30 s windows at a 25 s stride
    if args.precision == "bf16" and not args.graph and not args.no_extra_workloads:
        torch.cuda.empty_cache()
        pipe1 = wb.Pipeline(dims, stem, enc, 1, wb.PRESET_BF16)
        audio1 = audio[:synthetic.CHUNK_SAMPLES]
        wb.profile_begin()
        pipe1(audio1)
        torch.cuda.synchronize()
        launches1 = sum(n for _, n in wb.profile_end().values())
        graph1 = pipe1.capture(audio1)
        for _ in range(args.warmup):
            graph1.replay()
        torch.cuda.synchronize()
        n1 = 10 * args.steps
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        sampler = ClockSampler(gpu_uuid(torch, local))
        time.sleep(0.3)
        flush.zero_()
        ev1[0].record(stream)
        for _ in range(n1):
            graph1.replay()
        ev1[1].record(stream)
        torch.cuda.synchronize()
        clocks1 = sampler.stop()
        if wb.check_device_error() != 0:
            raise RuntimeError("device error in the batch-1 graph replays")
        ms1 = ev1[0].elapsed_time(ev1[1]) / n1
        line["batch1_graph"] = {
            "workload": "whisper large-v3 encoder hot path, batch 1 (one 30 s chunk), bf16, the three calls "
                        "replayed from one CUDA graph, back to back (weights ~1.27 GB, larger than L2)",
            "value": round(world * CHUNK_S / (ms1 / 1000.0), 2), "unit": UNIT, "ms_per_chunk": round(ms1, 4),
            "replays": n1, "gpu_launches_per_replay": launches1, "clocks": clocks1}
        del graph1, pipe1
        torch.cuda.empty_cache()

        stride, per = 400000, 36
        x_long = synthetic.long_audio(synthetic.SEED_LONGFORM)
        n_win = 1 + max(0, -(-(len(x_long) - synthetic.CHUNK_SAMPLES) // stride))
        xd = torch.from_numpy(x_long).cuda()
        pipe36 = wb.Pipeline(dims, stem, enc, per, wb.PRESET_BF16)

        def longform():
            for i in range(0, n_win, per):
                pipe36(xd[i * stride:], chunk_stride=stride, n_chunks=min(per, n_win - i))
        for _ in range(2):
            longform()
        torch.cuda.synchronize()
        reps = max(3, args.steps // 3)
        sampler = ClockSampler(gpu_uuid(torch, local))
        time.sleep(0.3)
        t_long = []
        for _ in range(reps):
            flush.zero_()
            ev1[0].record(stream)
            longform()
            ev1[1].record(stream)
            torch.cuda.synchronize()
            t_long.append(ev1[0].elapsed_time(ev1[1]))
        clocks_l = sampler.stop()
        if wb.check_device_error() != 0:
            raise RuntimeError("device error in the long-form runs")
        ms_l = statistics.median(t_long)
        audio_s = len(x_long) / float(synthetic.SAMPLE_RATE)
        line["longform"] = {
            "workload": (f"45 min of synthetic audio ({len(x_long)} samples, tone mix re-drawn every 10 s), "
                         f"{n_win} windows of 30 s at a 25 s stride, encoded in batches of {per} through the same "
                         "three calls, bf16, audio resident on the device (the batch-32 weights; throughput does "
                         "not depend on weight values)"),
            "value": round(world * audio_s / (ms_l / 1000.0), 2), "unit": UNIT, "ms": round(ms_l, 3),
            "windows": n_win, "reps": reps, "clocks": clocks_l}
        del pipe36, xd
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, parts = oracle_chunk_seconds(dims, seed)
        line["cpu_baseline"] = {
            "value": round(CHUNK_S / t, 5), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "host": cpu_info(),
            "sample": ("1 chunk of 30 s through the float64 oracle's log-mel, conv stem, 1 of 32 layers and one "
                       "LayerNorm; per-chunk time extrapolated to 32 layers"),
            "parts_s": {k: round(v, 3) for k, v in parts.items()}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
