"""Pins of the oracle's E4M3 codec: exhaustive over all 256 codes and all
midpoints, against torch's float8_e4m3fn type and the format's closed forms.  CPU only."""
import json
import os

import numpy as np
import torch

from oracle import fp8

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert (nan == np.isnan(got)).all() and nan.sum() == 2          # 0x7F and 0xFF
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert fp8.e4m3_decode(0x7E) == GOLDEN["e4m3_saturation"]["value"]
    assert fp8.e4m3_decode(0x01) == 2.0 ** -9 and fp8.e4m3_decode(0x08) == 2.0 ** -6


def test_encode_roundtrips_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_midpoints_round_to_even_code():
    vals = fp8.e4m3_decode(np.arange(0x7F))
    for c in range(0x7E):
        mid = 0.5 * (vals[c] + vals[c + 1])
        even = c if c % 2 == 0 else c + 1
        assert fp8.e4m3_encode(mid) == even
        assert fp8.e4m3_encode(-mid) == even | 0x80
        eps = (vals[c + 1] - vals[c]) * 1e-3
        assert fp8.e4m3_encode(mid - eps) == c and fp8.e4m3_encode(mid + eps) == c + 1


def test_encode_matches_torch_in_range():
    x = np.random.default_rng(0).normal(0, 60, size=200000).astype(np.float32)
    x = x[np.abs(x) < 440]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.e4m3_encode(x), ref)


def test_saturation_and_specials():
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e30, np.inf])
    assert (fp8.e4m3_encode(big) == 0x7E).all()
    assert (fp8.e4m3_encode(-big) == 0xFE).all()
    assert fp8.e4m3_encode(np.nan) == 0x7F
    assert fp8.e4m3_encode(0.0) == 0x00 and fp8.e4m3_encode(-0.0) == 0x80
    assert fp8.e4m3_encode(2.0 ** -10) == 0x00                 # tie between 0 and 2^-9 -> even
    assert fp8.e4m3_encode(1.5 * 2.0 ** -9) == 0x02            # tie between codes 1 and 2 -> even


def test_quantize_recipe():
    x = np.random.default_rng(1).normal(size=(300, 64)).astype(np.float32)
    x[5, 7] = -9.0                                             # the absmax element
    q, s = fp8.quantize(x)
    assert s == np.float32(9.0) / np.float32(448.0)
    assert q[5, 7] == 0xFE                                     # -448
    assert np.abs(fp8.e4m3_decode(q)).max() <= 448.0
    rel = np.abs(fp8.dequantize(q, s) - x) / np.maximum(np.abs(x), 1e-3)
    assert rel[np.abs(x) > 0.2].max() <= 2.0 ** -4 + 1e-6     # 3 mantissa bits: half-ulp <= 1/16
    q0, s0 = fp8.quantize(np.zeros(10, np.float32))
    assert s0 == 1.0 and (q0 == 0).all()


def test_e5m2_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = fp8.e5m2_decode(codes)
    assert (np.isnan(ref) == np.isnan(got)).all()
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert fp8.e5m2_decode(0x7B) == 57344.0 and fp8.e5m2_decode(0x7C) == np.inf


def test_e5m2_encode_roundtrip_midpoints_and_saturation():
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7C], dtype=np.uint8)
    np.testing.assert_array_equal(fp8.e5m2_encode(fp8.e5m2_decode(codes)), codes)
    vals = fp8.e5m2_decode(np.arange(0x7C))
    for c in range(0x7B):
        mid = 0.5 * (vals[c] + vals[c + 1])
        assert fp8.e5m2_encode(mid) == (c if c % 2 == 0 else c + 1)
    assert (fp8.e5m2_encode(np.array([57344.0, 60000.0, 1e9, np.inf])) == 0x7B).all()
    x = np.random.default_rng(2).normal(0, 3000, 100000).astype(np.float32)
    x = x[np.abs(x) < 57000]
    np.testing.assert_array_equal(fp8.e5m2_encode(x), torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy())


# --- bfloat16 storage rounding (the value an E4M3 site quantises) -----------------------------------

def _bits_to_f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_round_bf16_matches_torch_over_all_exponents():
    # float32 inputs are rounded once by both sides, so torch's cast is an independent reference
    rng = np.random.default_rng(3)
    mant = rng.integers(0, 1 << 23, size=400000, dtype=np.uint32)
    expo = rng.integers(0, 255, size=400000, dtype=np.uint32)          # every biased exponent incl. 0
    sign = rng.integers(0, 2, size=400000, dtype=np.uint32) << 31
    x = _bits_to_f32(sign | (expo << 23) | mant)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.round_bf16(x), ref)


def test_round_bf16_ties_go_to_the_even_significand():
    # low 16 bits exactly 0x8000: halfway between two bf16 values
    hi = np.arange(0x3F80, 0x3F90, dtype=np.uint32)                     # 1.0 .. 1.0 + 15 * 2^-7
    ties = _bits_to_f32((hi << 16) | 0x8000)
    expect = _bits_to_f32(((hi + (hi & 1)) << 16)).astype(np.float64)   # odd rounds up, even stays
    np.testing.assert_array_equal(fp8.round_bf16(ties), expect)
    np.testing.assert_array_equal(fp8.round_bf16(-ties), -expect)
    ref = torch.from_numpy(ties).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.round_bf16(ties), ref)
    # one unit past the tie rounds away from it whatever the parity
    np.testing.assert_array_equal(fp8.round_bf16(_bits_to_f32((hi << 16) | 0x8001)),
                                  _bits_to_f32((hi + 1) << 16).astype(np.float64))


def test_round_bf16_rounds_the_exact_value_once():
    # 1 + 2^-8 + 2^-40 lies just above the tie between 1 and 1 + 2^-7: nearest is 1 + 2^-7.
    # Rounding it to float32 first would land exactly on the tie and then go to the even 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert fp8.round_bf16(x) == 1.0 + 2.0 ** -7
    assert fp8.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert fp8.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6       # tie, odd -> up to even


def test_round_bf16_subnormals_overflow_and_specials():
    tiny = 2.0 ** -133                                                    # smallest bf16 subnormal
    assert fp8.round_bf16(tiny) == tiny and fp8.round_bf16(0.5 * tiny) == 0.0    # tie -> even (0)
    assert fp8.round_bf16(0.75 * tiny) == tiny and fp8.round_bf16(1.5 * tiny) == 2 * tiny
    assert fp8.round_bf16(2.0 ** -126 - tiny) == 2.0 ** -126 - tiny       # largest subnormal is exact
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127                                  # largest finite bf16
    assert fp8.round_bf16(big) == big
    assert fp8.round_bf16(big + 2.0 ** 119) == np.inf                     # halfway to 2^128: tie -> even -> inf
    assert fp8.round_bf16(big + 2.0 ** 118) == big
    assert fp8.round_bf16(-np.inf) == -np.inf and np.isnan(fp8.round_bf16(np.nan))
    assert np.signbit(fp8.round_bf16(-0.0)) and fp8.round_bf16(-0.0) == 0.0
    assert np.isnan(fp8.round_bf16(_bits_to_f32(0x7F800001)))            # a NaN payload stays NaN


def test_activation_site_matches_torch_dtypes():
    # bf16 storage then per-tensor E4M3 (scale amax / 448), rebuilt from torch's bfloat16 and
    # float8_e4m3fn casts; float32-valued input so that both sides round it once
    rng = np.random.default_rng(4)
    a = (rng.normal(size=(64, 96)) * 3.0).astype(np.float32)
    got = fp8.fake_quantize(fp8.round_bf16(a))
    t = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32)
    amax = t.abs().max()
    inv = torch.tensor(448.0, dtype=torch.float32) / amax
    codes = (t * inv).to(torch.float8_e4m3fn)
    ref = codes.to(torch.float64) * (amax / torch.tensor(448.0, dtype=torch.float32)).to(torch.float64)
    np.testing.assert_array_equal(got, ref.numpy())


# --- E5M2 per-tensor scale recipe ----------------------------------------------------------------

def test_quantize_e5m2_scale_recipe():
    rng = np.random.default_rng(5)
    x = (rng.normal(size=(200, 64)) * 40.0).astype(np.float32)
    x[3, 9] = -1234.5                                                     # the absmax element
    q, s = fp8.quantize_e5m2(x)
    assert s == np.float32(1234.5) / np.float32(57344.0)                 # dequantisation scale
    assert q[3, 9] == 0xFB                                                # -57344, the largest finite code
    qn, sn = fp8.quantize_e5m2(-x)
    assert sn == s and np.array_equal(qn, q ^ 0x80)                       # sign symmetry
    deq = fp8.e5m2_decode(q) * np.float64(s)
    big = np.abs(x) > 1e-3 * 1234.5                                       # away from the subnormal codes
    rel = np.abs(deq - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -3 * (1 + 1e-6)                            # 2 significand bits: half-ulp <= 1/8
    q0, s0 = fp8.quantize_e5m2(np.zeros((4, 4), np.float32))
    assert s0 == 1.0 and (q0 == 0).all()


def test_quantize_e5m2_matches_torch_dtype():
    # the same recipe rebuilt from torch's float8_e5m2 cast
    x = (np.random.default_rng(6).normal(size=(128, 80)) * 0.3).astype(np.float32)
    q, s = fp8.quantize_e5m2(x)
    t = torch.from_numpy(x)
    amax = t.abs().max()
    ref = (t * (torch.tensor(57344.0) / amax)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q, ref)
    assert s == (amax / torch.tensor(57344.0)).item()
