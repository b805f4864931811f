"""FP8 E4M3 codec and per-tensor absmax scaling (oracle; test infrastructure only).

The whisper-blaze showcase site, "The Solution" (fp8_quantize.cu card:
per-tensor scale, amax) and "Learnings" (E4M3 saturates at 448; scales come
from activation maxima), and the PyPI page, "Direct Kernel API"
(quantise_e4m3 returns codes and a per-tensor scale).

Format (OCP 8-bit floating point, E4M3 "fn" variant): sign bit, 4 exponent
bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
m * 2^-9; S.1111.111 is NaN; there are no infinities; the largest finite
magnitude is 1.75 * 2^8 = 448.

Reading where the pages are silent: rounding is to nearest, ties to the even
code; magnitudes above 448 (and infinities) saturate to 448; NaN stays NaN.
The scaling recipe (taken in float32, the precision the GPU path uses):
    amax  = max |x|                  (float32)
    scale = amax / 448               (dequantisation scale; 1 when amax == 0)
    inv   = 448 / amax               (1 when amax == 0)
    code  = e4m3(float32(x) * inv)   (one float32 multiply, then RNE + saturate)
Dequantisation is decode(code) * scale.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """Exact float64 value of each 8-bit code."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((c & 0x7F) == NAN_CODE, np.nan, val)
    return sign * val


# Non-negative finite values in code order 0x00 .. 0x7E (monotonic in the code).
_POS_VALUES = e4m3_decode(np.arange(0x7F))


def e4m3_encode(x) -> np.ndarray:
    """Round each value to E4M3: nearest, ties to even code, saturate to +-448."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    hi = np.searchsorted(_POS_VALUES, ax, side="left")      # first value >= ax
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = ax - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - ax
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(ax >= E4M3_MAX, 0x7E, code)               # saturate (incl. +inf)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), NAN_CODE, code)
    return code.astype(np.uint8)


def absmax_scale(x):
    """(amax, scale, inv) of the per-tensor recipe, all float32."""
    amax = np.float32(np.max(np.abs(np.asarray(x, dtype=np.float32)))) if np.size(x) else np.float32(0)
    if amax == 0:
        return amax, np.float32(1.0), np.float32(1.0)
    return amax, np.float32(amax / np.float32(E4M3_MAX)), np.float32(np.float32(E4M3_MAX) / amax)


def quantize(x):
    """Per-tensor E4M3 quantisation: (codes uint8, scale float32)."""
    x32 = np.asarray(x, dtype=np.float32)
    _, scale, inv = absmax_scale(x32)
    return e4m3_encode((x32 * inv).astype(np.float32)), scale


def dequantize(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) * np.float64(scale)


def round_bf16(x) -> np.ndarray:
    """Round each value once to bfloat16 and return the results as float64.

    An activation is stored as bf16 before it is quantised, so the quantisation
    decision is taken on the bf16 value.  bfloat16 (the format of the Google
    Brain float and of the Arm / Intel ISA extensions that adopted it): sign, the
    8 exponent bits of IEEE binary32, 7 stored significand bits, so 8
    significant bits, subnormals spaced 2^-133 apart below 2^-126, largest
    finite magnitude (2 - 2^-7) * 2^127.  Rounding is to nearest, ties to the
    even significand, applied to the exact input value (no intermediate
    float32 rounding); magnitudes that round past the largest finite value
    become infinities; +-inf and NaN pass through.
    """
    with np.errstate(over="ignore", invalid="ignore"):
        x = np.asarray(x, dtype=np.float64)
        m, e = np.frexp(x)                                   # x = m * 2^e, 0.5 <= |m| < 1
        normal = np.rint(m * 256.0) * np.exp2(e.astype(np.float64) - 8.0)   # 8 significant bits
        sub = np.rint(x * 2.0 ** 133) * 2.0 ** -133                         # fixed spacing below 2^-126
        r = np.where(np.abs(x) < 2.0 ** -126, sub, normal)
        r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def fake_quantize(x) -> np.ndarray:
    """dequantize(quantize(x)): the value an E4M3 operand with one per-tensor scale carries."""
    codes, scale = quantize(np.asarray(x, dtype=np.float32))
    return dequantize(codes, scale)


# --- E5M2 ----------------------------------------------------------------------------------------
# The showcase site, "The Solution" (fp8_quantize.cu card: casts for both E4M3 and E5M2, "more
# range") and "The Approach" (aggressive_fp8 switches cross-attention activations to E5M2).
# Format (OCP 8-bit floating point, E5M2): sign, 5 exponent bits with bias 15, 2 mantissa bits;
# exponent field 0 encodes subnormals m * 2^-16; exponent 31 encodes inf (m = 0) and NaN;
# the largest finite magnitude is 1.75 * 2^15 = 57344.  Rounding reading as for E4M3: nearest,
# ties to the even code, magnitudes above 57344 (and infinities) saturate to +-57344.

E5M2_MAX = 57344.0


def e5m2_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = (c & 0x3).astype(np.float64)
    val = np.where(e == 0, m / 4.0 * 2.0 ** -14, (1.0 + m / 4.0) * np.exp2(e.astype(np.float64) - 15.0))
    val = np.where(e == 31, np.where(m == 0, np.inf, np.nan), val)
    return sign * val


_POS_E5M2 = e5m2_decode(np.arange(0x7C))        # finite non-negative values, codes 0x00 .. 0x7B


def e5m2_encode(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    hi = np.minimum(np.searchsorted(_POS_E5M2, ax, side="left"), len(_POS_E5M2) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = ax - _POS_E5M2[lo]
    d_hi = _POS_E5M2[hi] - ax
    code = np.where((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)), hi, lo)
    code = np.where(ax >= E5M2_MAX, 0x7B, code)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_e5m2(x):
    """Per-tensor E5M2: scale = amax / 57344, code = e5m2(float32(x) * (57344 / amax))."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    if amax == 0:
        return e5m2_encode(x32), np.float32(1.0)
    inv = np.float32(np.float32(E5M2_MAX) / amax)
    return e5m2_encode((x32 * inv).astype(np.float32)), np.float32(amax / np.float32(E5M2_MAX))
