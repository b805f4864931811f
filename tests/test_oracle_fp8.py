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
