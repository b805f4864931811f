"""Conv stem and pre-LN encoder layers in float64 (oracle; test infrastructure only).

The whisper-blaze pages name the components (the showcase site, "The
Solution": workhorse GEMM, fused encoder self-attention that never writes the
score matrix, fused residual + LayerNorm; the PyPI page, "Direct Kernel API":
LayerNorm eps 1e-5, and the feature list: 162 LayerNorms in the model, i.e.
32*2 + 1 = 65 in the encoder) but never write out their equations.  The
oracle takes the plainest reading, the standard published Whisper encoder:

  stem   y1 = GELU(conv1d(logmel; C->d, k3, stride 1, pad 1))
         x0 = GELU(conv1d(y1;     d->d, k3, stride 2, pad 1)) + PE
  layer  a = LN1(h); q = a Wq^T + bq; k = a Wk^T; v = a Wv^T + bv
         h += concat_h(softmax(q_h k_h^T / sqrt(64)) v_h) Wo^T + bo
         h += GELU(LN2(h) W1^T + b1) W2^T + b2
  final  out = LN_post(h)

GELU is the exact erf form; convolutions are cross-correlations with zero
padding; LayerNorm uses the biased variance.  Attention has no mask (the
encoder is non-causal) and runs over all 1500 positions.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

LN_EPS = 1e-5


def gelu(x):
    """x * Phi(x) with the exact normal CDF."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def sinusoids(n_pos: int, d: int, max_timescale: float = 10000.0) -> np.ndarray:
    """Whisper's positional table: sin in the first d/2 columns, cos in the rest.

    Column i < d/2 uses frequency exp(-i * ln(max_timescale) / (d/2 - 1)).
    """
    half = d // 2
    inc = math.log(max_timescale) / (half - 1)
    inv = np.exp(-inc * np.arange(half, dtype=np.float64))
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.sin(ang), np.cos(ang)], axis=1)


def conv1d_k3(x: np.ndarray, w: np.ndarray, b: np.ndarray, stride: int) -> np.ndarray:
    """Cross-correlation with kernel 3, zero padding 1.

    x [C_in, T_in], w [C_out, C_in, 3], b [C_out] -> [C_out, T_out],
    out[c, t] = b[c] + sum_{ci, j} w[c, ci, j] * x[ci, stride*t + j - 1].
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    c_in, t_in = x.shape
    xp = np.zeros((c_in, t_in + 2))
    xp[:, 1:-1] = x
    t_out = (t_in + 2 - 3) // stride + 1
    out = np.zeros((w.shape[0], t_out)) + np.asarray(b, dtype=np.float64)[:, None]
    for j in range(3):
        cols = xp[:, j + stride * np.arange(t_out)]
        out += w[:, :, j] @ cols
    return out


def conv_stem(logmel: np.ndarray, weights: dict) -> np.ndarray:
    """log-mel [C, 3000] -> x0 [1500, d]: two GELU convolutions plus positions."""
    y1 = gelu(conv1d_k3(logmel, weights["conv1_w"], weights["conv1_b"], 1))
    y2 = gelu(conv1d_k3(y1, weights["conv2_w"], weights["conv2_b"], 2))
    x0 = y2.T
    return x0 + sinusoids(x0.shape[0], x0.shape[1])


def layer_norm(x: np.ndarray, g, b, eps: float = LN_EPS) -> np.ndarray:
    """(x - mean) / sqrt(var + eps) * g + b over the last axis, biased variance."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(g, np.float64) + np.asarray(b, np.float64)


def rms_norm(x: np.ndarray, g, eps: float = LN_EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis (the PyPI page, "Direct Kernel API": rmsnorm_fused)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * np.asarray(g, np.float64)


def softmax(s: np.ndarray) -> np.ndarray:
    """Row softmax (max subtracted first, which leaves the value unchanged)."""
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int) -> np.ndarray:
    """Multi-head softmax attention without a mask: [T, d] x3 -> [T, d]."""
    T, d = q.shape
    hd = d // n_heads
    out = np.empty((T, d))
    for h in range(n_heads):
        sl = slice(h * hd, (h + 1) * hd)
        p = softmax(q[:, sl] @ k[:, sl].T / math.sqrt(hd))
        out[:, sl] = p @ v[:, sl]
    return out


def encoder_layer(h: np.ndarray, L: dict, n_heads: int, fp8_sites=()) -> np.ndarray:
    """One pre-LN Whisper encoder layer on a [T, d] float64 residual stream.

    ``fp8_sites`` names the layer sites ("qkv", "out", "ffn") whose GEMMs take
    E4M3 operands (the whisper-blaze showcase site, "The Approach": mixed_fp8
    puts encoder_attn_qkv and encoder_ffn in E4M3 for weights and activations,
    encoder_attn_out stays 16-bit).  Each operand then carries one per-tensor
    absmax scale: the fused [3d, d] QKV weight, W1, W2 and W_o as matrices, and
    each activation over the whole [T, k] operand after it is stored as bf16.
    Everything else stays float64.
    """
    from . import fp8 as q8
    f64 = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    act = (lambda a: q8.fake_quantize(q8.round_bf16(a)))  # noqa: E731
    wgt = q8.fake_quantize
    d = h.shape[1]
    a = layer_norm(h, L["ln1_g"], L["ln1_b"])
    w_qkv = np.concatenate([f64(L["wq"]), f64(L["wk"]), f64(L["wv"])])
    if "qkv" in fp8_sites:
        qkv = act(a) @ wgt(w_qkv).T
    else:
        qkv = a @ w_qkv.T
    q = qkv[:, :d] + f64(L["bq"])
    k = qkv[:, d:2 * d]
    v = qkv[:, 2 * d:] + f64(L["bv"])
    o = attention(q, k, v, n_heads)
    if "out" in fp8_sites:
        h = h + act(o) @ wgt(L["wo"]).T + f64(L["bo"])
    else:
        h = h + o @ f64(L["wo"]).T + f64(L["bo"])
    f = layer_norm(h, L["ln2_g"], L["ln2_b"])
    if "ffn" in fp8_sites:
        g = gelu(act(f) @ wgt(L["w1"]).T + f64(L["b1"]))
        h = h + act(g) @ wgt(L["w2"]).T + f64(L["b2"])
    else:
        h = h + gelu(f @ f64(L["w1"]).T + f64(L["b1"])) @ f64(L["w2"]).T + f64(L["b2"])
    return h


MIXED_FP8 = ("qkv", "ffn")


def encoder(x0: np.ndarray, weights: dict, n_heads: int, layer_begin: int = 0,
            layer_end: int | None = None, final_ln: bool = True, capture: list | None = None,
            fp8_sites=()):
    """Layers [layer_begin, layer_end) on x0 [T, d], then optionally LN_post.

    If ``capture`` is a list, the residual stream after every layer is appended.
    ``fp8_sites`` as in encoder_layer (MIXED_FP8 for the mixed_fp8 preset).
    """
    layers = weights["layers"]
    if layer_end is None:
        layer_end = len(layers)
    h = np.asarray(x0, dtype=np.float64)
    for i in range(layer_begin, layer_end):
        h = encoder_layer(h, layers[i], n_heads, fp8_sites)
        if capture is not None:
            capture.append(h)
    if final_ln:
        h = layer_norm(h, weights["ln_post_g"], weights["ln_post_b"])
    return h


def forward(chunk: np.ndarray, weights: dict, n_mels: int, n_heads: int, **kw) -> np.ndarray:
    """Audio chunk [480000] -> encoder output [1500, d] (log-mel, stem, layers, LN_post)."""
    from . import frontend
    return encoder(conv_stem(frontend.log_mel(chunk, n_mels), weights), weights, n_heads, **kw)


def cross_kv(enc_out: np.ndarray, layers: list) -> list:
    """Decoder cross-attention keys and values of the encoder output, one (K, V) pair per decoder layer.

    The showcase site, "The Approach" (decoder_cross_attn site) and "The Solution" (decoder
    cross-attention is one of the three attention patterns): the decoder attends to the
    encoder output through its own key / value projections; Whisper's key projection has no
    bias.  K = enc_out Wk^T, V = enc_out Wv^T + bv, enc_out [T, d].
    """
    f64 = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    e = f64(enc_out)
    return [(e @ f64(L["wk"]).T, e @ f64(L["wv"]).T + f64(L["bv"])) for L in layers]
