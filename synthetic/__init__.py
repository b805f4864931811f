"""Seeded synthetic inputs for the Whisper large-v3 encoder hot path.

This module is shared by the CPU oracle tests, the GPU parity tests, the smoke
check and the benchmark.  It only DRAWS inputs (audio samples and random-init
weights); it holds no step of the method's arithmetic.  Both the oracle and
the CUDA path consume exactly the values it returns.

Audio (the whisper-blaze PyPI page, "Quick Start": float32 mono at 16 kHz):
  one 30 s chunk = 480000 samples; sum of 3 zero-phase sines with frequencies
  drawn U(100, 4000) Hz and amplitudes U(0.1, 0.3), plus N(0, sigma=0.01)
  noise.  Draw order per chunk: 3 frequencies, 3 amplitudes, 480000 noise
  values, from numpy's PCG64 ``default_rng(seed)``.  The sum is formed in
  float64 and stored as float32.

Long-form audio (45 min): amplitudes drawn once, then per 10 s segment
  (160000 samples) 3 fresh frequencies followed by that segment's noise; time
  n is global, so the sines keep their phase across segments.

Weights (random init, no trained checkpoint): Linear weights, conv weights
  and biases ~N(0, 0.02); LayerNorm gamma = 1 + N(0, 0.02), beta = N(0, 0.02).
  Drawn in a fixed order (stem, then each layer, then the final LayerNorm) and
  rounded to the configuration's storage dtype ("f32" or "bf16" with
  round-to-nearest-even).  Arrays are returned as float32 holding exactly the
  rounded values.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SAMPLE_RATE = 16000
CHUNK_SAMPLES = 480000          # 30 s at 16 kHz
LONG_SEGMENT = 160000           # long-form: frequencies re-drawn every 10 s


@dataclasses.dataclass(frozen=True)
class Dims:
    """Encoder shape: mel bins, model width, heads, layers, FFN width."""
    n_mels: int
    d_model: int
    n_heads: int
    n_layers: int
    d_ffn: int

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads


TINY = Dims(n_mels=80, d_model=384, n_heads=6, n_layers=1, d_ffn=1536)
LARGE_V3 = Dims(n_mels=128, d_model=1280, n_heads=20, n_layers=32, d_ffn=5120)

# Base seeds of the five workloads (tiny; large-v3 batch 1; batch 32 bf16 and
# mixed-fp8 share inputs; long-form 45 min).
SEED_TINY = 0
SEED_LARGE_B1 = 1000
SEED_LARGE_B32 = 2000
SEED_LONGFORM = 3000


def tone_chunk(seed: int, n: int = CHUNK_SAMPLES) -> np.ndarray:
    """One chunk of the 3-sine + noise test signal, float32 [n]."""
    rng = np.random.default_rng(seed)
    freqs = rng.uniform(100.0, 4000.0, 3)
    amps = rng.uniform(0.1, 0.3, 3)
    noise = rng.normal(0.0, 0.01, n)
    t = np.arange(n, dtype=np.float64)
    x = noise.copy()
    for f, a in zip(freqs, amps):
        x += a * np.sin(2.0 * np.pi * f * t / SAMPLE_RATE)
    return x.astype(np.float32)


def tone_batch(base_seed: int, batch: int, n: int = CHUNK_SAMPLES) -> np.ndarray:
    """``batch`` independent chunks, chunk b seeded with base_seed + b: float32 [batch, n]."""
    return np.stack([tone_chunk(base_seed + b, n) for b in range(batch)])


def long_audio(seed: int, n_samples: int = 43_200_000) -> np.ndarray:
    """Long-form tone mix: frequencies re-drawn every 10 s, float32 [n_samples]."""
    rng = np.random.default_rng(seed)
    amps = rng.uniform(0.1, 0.3, 3)
    out = np.empty(n_samples, dtype=np.float32)
    for s0 in range(0, n_samples, LONG_SEGMENT):
        s1 = min(n_samples, s0 + LONG_SEGMENT)
        freqs = rng.uniform(100.0, 4000.0, 3)
        noise = rng.normal(0.0, 0.01, s1 - s0)
        t = np.arange(s0, s1, dtype=np.float64)
        x = noise
        for f, a in zip(freqs, amps):
            x = x + a * np.sin(2.0 * np.pi * f * t / SAMPLE_RATE)
        out[s0:s1] = x.astype(np.float32)
    return out


def silence(n: int = CHUNK_SAMPLES) -> np.ndarray:
    return np.zeros(n, dtype=np.float32)


def half_silence(seed: int, n: int = CHUNK_SAMPLES) -> np.ndarray:
    """First half a tone chunk, second half exact zeros (drives the log clamp)."""
    x = tone_chunk(seed, n)
    x[n // 2:] = 0.0
    return x


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype ("f32" or "bf16", RNE)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype != "bf16":
        raise ValueError(dtype)
    import torch   # a storage-format conversion, not part of the method
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()


def _normal(rng, shape, std=0.02):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


def encoder_weights(dims: Dims, seed: int, dtype: str = "bf16", n_layers: int | None = None) -> dict:
    """Random-init encoder weights in the HF Whisper layout.

    Returns {"conv1_w": [d, C, 3], "conv1_b": [d], "conv2_w": [d, d, 3],
    "conv2_b": [d], "layers": [dict per layer], "ln_post_g", "ln_post_b"}.
    Per layer: ln1_g, ln1_b, wq [d,d], bq, wk [d,d], wv [d,d], bv, wo [d,d],
    bo, ln2_g, ln2_b, w1 [F,d], b1 [F], w2 [d,F], b2 [d].  The k projection
    has no bias.  All float32 arrays holding values of ``dtype``.  With
    ``n_layers`` < dims.n_layers only the first layers are drawn (identical to
    the full draw's first layers) and the final LayerNorm is omitted.
    """
    rng = np.random.default_rng(seed)
    d, C, F = dims.d_model, dims.n_mels, dims.d_ffn
    r = lambda a: round_to(a, dtype)  # noqa: E731
    w = {}
    w["conv1_w"] = r(_normal(rng, (d, C, 3)))
    w["conv1_b"] = r(_normal(rng, (d,)))
    w["conv2_w"] = r(_normal(rng, (d, d, 3)))
    w["conv2_b"] = r(_normal(rng, (d,)))
    layers = []
    count = dims.n_layers if n_layers is None else n_layers
    for _ in range(count):
        L = {}
        L["ln1_g"] = r(1.0 + _normal(rng, (d,)))
        L["ln1_b"] = r(_normal(rng, (d,)))
        L["wq"] = r(_normal(rng, (d, d)))
        L["bq"] = r(_normal(rng, (d,)))
        L["wk"] = r(_normal(rng, (d, d)))
        L["wv"] = r(_normal(rng, (d, d)))
        L["bv"] = r(_normal(rng, (d,)))
        L["wo"] = r(_normal(rng, (d, d)))
        L["bo"] = r(_normal(rng, (d,)))
        L["ln2_g"] = r(1.0 + _normal(rng, (d,)))
        L["ln2_b"] = r(_normal(rng, (d,)))
        L["w1"] = r(_normal(rng, (F, d)))
        L["b1"] = r(_normal(rng, (F,)))
        L["w2"] = r(_normal(rng, (d, F)))
        L["b2"] = r(_normal(rng, (d,)))
        layers.append(L)
    w["layers"] = layers
    if count == dims.n_layers:
        w["ln_post_g"] = r(1.0 + _normal(rng, (d,)))
        w["ln_post_b"] = r(_normal(rng, (d,)))
    return w


def cross_kv_weights(dims: Dims, seed: int, n_layers: int, dtype: str = "bf16") -> list:
    """Random-init decoder cross-attention projections per decoder layer: wk, wv [d, d], bv [d]."""
    rng = np.random.default_rng(seed)
    d = dims.d_model
    out = []
    for _ in range(n_layers):
        out.append({"wk": round_to(_normal(rng, (d, d)), dtype), "wv": round_to(_normal(rng, (d, d)), dtype),
                    "bv": round_to(_normal(rng, (d,)), dtype)})
    return out


def gemm_operands(seed: int, m: int, n: int, k: int, lo: int = -3, hi: int = 3):
    """Small-integer GEMM operands (exact in bf16 and E4M3), float32 arrays."""
    rng = np.random.default_rng(seed)
    a = rng.integers(lo, hi + 1, (m, k)).astype(np.float32)
    b = rng.integers(lo, hi + 1, (n, k)).astype(np.float32)
    return a, b
