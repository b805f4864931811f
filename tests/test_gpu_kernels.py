"""Kernel-level parity of libwb against the oracle, through the C ABI (GPU).

GEMMs on small-integer operands are bit-exact (bf16 and E4M3 hold small
integers exactly and the fp32 accumulation of the products is exact); the
other kernels are compared with the oracle's float64 results on seeded inputs
at sizes that span several tiles plus a ragged tail."""
import numpy as np
import pytest
import torch

from conftest import rel_l2, to_np
from oracle import encoder as oenc
from oracle import fp8 as ofp8
import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(DEV).to(torch.bfloat16)


def _f32(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(DEV)


@pytest.mark.parametrize("M,N,K", [(300, 256, 320), (128, 384, 64), (1000, 1152, 384), (1, 32, 8), (4100, 512, 1280)])
def test_linear_bf16_small_integers_bit_exact(wb, M, N, K):
    a, w = synthetic.gemm_operands(M * 7 + N, M, N, K, -1, 1)
    rng = np.random.default_rng(K)
    bias = rng.integers(-4, 5, N).astype(np.float32)
    resid = rng.integers(-4, 5, (M, N)).astype(np.float32)
    ref = a.astype(np.int64) @ w.astype(np.int64).T + bias.astype(np.int64) + resid.astype(np.int64)
    assert np.abs(ref).max() <= 256                       # representable exactly in bf16
    out = wb.linear(_bf16(a), _bf16(w), bias=_f32(bias), resid=_bf16(resid))
    assert wb.check_device_error() == 0
    np.testing.assert_array_equal(to_np(out), ref.astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(25600, 1152, 64), (48000, 1280, 128)])
def test_linear_bf16_wide_tiles_bit_exact(wb, M, N, K):
    # M large enough that the 256-column tiles are chosen (ragged last column tile for N = 1152); the
    # small-M cases above run 128-column tiles
    a, w = synthetic.gemm_operands(M + N, M, N, K, -1, 1)
    rng = np.random.default_rng(N)
    bias = rng.integers(-4, 5, N).astype(np.float32)
    ref = a.astype(np.float64) @ w.astype(np.float64).T + bias      # small integers: exact in float64
    out = wb.linear(_bf16(a), _bf16(w), bias=_f32(bias), gelu=False)
    assert wb.check_device_error() == 0
    np.testing.assert_array_equal(to_np(out), ref)


@pytest.mark.parametrize("M,N,K", [(300, 256, 256), (257, 1280, 640)])
def test_linear_e4m3_small_integers_bit_exact(wb, M, N, K):
    a, w = synthetic.gemm_operands(5 * M + K, M, N, K, -2, 2)
    qa = torch.as_tensor(ofp8.e4m3_encode(a)).to(DEV)
    qw = torch.as_tensor(ofp8.e4m3_encode(w)).to(DEV)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    half = torch.full((1,), 0.5, dtype=torch.float32, device=DEV)
    out = wb.linear(qa, qw, scale_a=one, scale_w=half)
    ref = (a.astype(np.int64) @ w.astype(np.int64).T) * 0.5
    assert np.abs(ref).max() <= 256
    np.testing.assert_array_equal(to_np(out), ref)


def test_linear_gelu_bias_matches_oracle(wb):
    rng = np.random.default_rng(3)
    M, N, K = 700, 1536, 384
    a = synthetic.round_to(rng.normal(size=(M, K)).astype(np.float32), "bf16")
    w = synthetic.round_to((rng.normal(size=(N, K)) * 0.05).astype(np.float32), "bf16")
    b = rng.normal(size=N).astype(np.float32) * 0.1
    out = wb.linear(_bf16(a), _bf16(w), bias=_f32(b), gelu=True)
    ref = oenc.gelu(a.astype(np.float64) @ w.astype(np.float64).T + b)
    assert rel_l2(to_np(out), ref) < 4e-3


def test_fp8_gemm_matches_dequantized_operands(wb):
    # E4M3 GEMM vs an fp64 GEMM of the dequantised (exactly representable) operands
    rng = np.random.default_rng(4)
    M, N, K = 513, 768, 1024
    a = rng.normal(size=(M, K)).astype(np.float32)
    w = (rng.normal(size=(N, K)) * 0.02).astype(np.float32)
    qa, sa = wb.quantize_fp8(_bf16(a))
    qw, sw = wb.quantize_fp8(_bf16(w))
    out = wb.linear(qa, qw, scale_a=sa, scale_w=sw)
    da = ofp8.dequantize(qa.cpu().numpy(), sa.item())
    dw = ofp8.dequantize(qw.cpu().numpy(), sw.item())
    ref = da @ dw.T
    # the output is bf16: compare with the exact product rounded to bf16 (that
    # rounding alone is ~1.1e-3 relative L2, so it cannot be part of the budget)
    assert rel_l2(to_np(out), synthetic.round_to(ref.astype(np.float32), "bf16")) < 1e-3
    assert rel_l2(to_np(out), ref) < 2.5e-3


@pytest.mark.parametrize("n", [16, 4096 * 33 + 7, 1280 * 1500])
def test_quantize_fp8_bit_exact_vs_oracle_codec(wb, n):
    rng = np.random.default_rng(n)
    x = synthetic.round_to((rng.normal(size=n) * 3.0).astype(np.float32), "bf16")
    x[n // 3] = -11.5
    q, s = wb.quantize_fp8(_bf16(x))
    q_ref, s_ref = ofp8.quantize(x)
    assert s.item() == float(s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    y = wb.dequantize_fp8(q, s)
    np.testing.assert_array_equal(to_np(y), synthetic.round_to(ofp8.dequantize(q_ref, s_ref).astype(np.float32), "bf16"))


def test_quantize_zero_tensor_scale_one(wb):
    q, s = wb.quantize_fp8(torch.zeros(64, dtype=torch.bfloat16, device=DEV))
    assert s.item() == 1.0 and int(q.sum()) == 0


@pytest.mark.parametrize("d,rows", [(1280, 3001), (384, 1500), (512, 7)])
def test_layernorm_matches_oracle(wb, d, rows):
    rng = np.random.default_rng(d)
    x = synthetic.round_to(rng.normal(0.3, 2.0, size=(rows, d)).astype(np.float32), "bf16")
    r = synthetic.round_to(rng.normal(size=(rows, d)).astype(np.float32), "bf16")
    g = (1 + 0.1 * rng.normal(size=d)).astype(np.float32)
    b = (0.1 * rng.normal(size=d)).astype(np.float32)
    y, tot = wb.layernorm(_bf16(x), _f32(g), _f32(b), 1e-5, residual=_bf16(r), return_total=True)
    ref = oenc.layer_norm(x.astype(np.float64) + r, g, b)
    assert np.abs(to_np(y) - ref).max() < 0.02 * np.abs(ref).max() / 4
    assert rel_l2(to_np(y), ref) < 4e-3
    np.testing.assert_array_equal(to_np(tot), synthetic.round_to((x + r).astype(np.float32), "bf16"))
    y2 = wb.layernorm(_bf16(x), _f32(g), _f32(b), 1e-5)
    assert rel_l2(to_np(y2), oenc.layer_norm(x.astype(np.float64), g, b)) < 4e-3


@pytest.mark.parametrize("d,rows,rpi", [(1280, 3700, 1500), (384, 1500, 1500), (640, 301, 100), (128, 1, 1)])
def test_layernorm_e4m3_matches_two_step_path_and_oracle(wb, d, rows, rpi):
    rng = np.random.default_rng(d + rows)
    x = rng.normal(0.3, 2.0, size=(rows, d)).astype(np.float32)
    x[:, 5] *= 40.0                                    # an outlier feature, as in real activations
    x = synthetic.round_to(x, "bf16")                  # the oracle sees exactly the bf16 input
    g = (1 + 0.1 * rng.normal(size=d)).astype(np.float32)
    b = (0.1 * rng.normal(size=d)).astype(np.float32)
    q, amax, stats = wb.layernorm_e4m3(_bf16(x), _f32(g), _f32(b), 1e-5, rows_per_item=rpi)
    assert wb.check_device_error() == 0
    q, amax, stats = to_np(q).astype(np.uint8), to_np(amax), to_np(stats)
    y = wb.layernorm(_bf16(x), _f32(g), _f32(b), 1e-5)           # bf16 LayerNorm, then a per-item quantiser
    for i in range(0, rows, rpi):
        yi = y[i:i + rpi]
        qi, si = wb.quantize_fp8(yi)
        # same arithmetic; the row statistics are summed in another order, so a value on a rounding
        # boundary may land one bf16 / E4M3 step away
        a2 = np.abs(to_np(yi)).max()
        assert abs(amax[i // rpi] - a2) <= a2 * 2.0 ** -8
        q2 = to_np(qi).astype(np.uint8)
        diff = q[i:i + rpi] != q2
        assert diff.mean() < 1e-4
        assert np.all(np.abs(ofp8.e4m3_decode(q[i:i + rpi][diff]) - ofp8.e4m3_decode(q2[diff]))
                      <= 2.0 ** -3 * np.abs(ofp8.e4m3_decode(q2[diff])) + 2.0 ** -9)
        # against the float64 oracle: one E4M3 rounding (relative 2^-4) on top of bf16 LayerNorm accuracy
        ref = oenc.layer_norm(x[i:i + rpi].astype(np.float64), g, b)
        dec = ofp8.e4m3_decode(q[i:i + rpi]) * (amax[i // rpi] / 448.0)
        assert np.all(np.abs(dec - ref) <= 0.07 * np.abs(ref) + amax[i // rpi] / 448.0 * 2.0 ** -8)
    mu = x.astype(np.float64).mean(axis=1)
    rs = 1.0 / np.sqrt(x.astype(np.float64).var(axis=1) + 1e-5)
    np.testing.assert_allclose(stats[:, 0], mu, rtol=1e-4, atol=1e-4 * np.abs(x).max())
    np.testing.assert_allclose(stats[:, 1], rs, rtol=1e-4)


@pytest.mark.parametrize("B,T,H", [(1, 1500, 2), (2, 130, 3), (1, 64, 1), (1, 257, 2), (1, 1, 1), (1, 9, 1),
                                   (1, 127, 1), (1, 128, 2), (1, 129, 1), (2, 255, 1)])
def test_attention_matches_oracle(wb, B, T, H):
    rng = np.random.default_rng(T + H)
    d = 64 * H
    q, k, v = (synthetic.round_to(rng.normal(size=(B, T, d)).astype(np.float32), "bf16") for _ in range(3))
    out = to_np(wb.attention(_bf16(q), _bf16(k), _bf16(v), H))
    assert wb.check_device_error() == 0
    for b in range(B):
        ref = oenc.attention(q[b].astype(np.float64), k[b], v[b], H)
        assert rel_l2(out[b], ref) < 1e-2


def test_attention_peaked_scores(wb):
    # large-magnitude scores exercise the running-max rescale across key tiles
    rng = np.random.default_rng(11)
    B, T, H = 1, 700, 1
    q = synthetic.round_to((rng.normal(size=(B, T, 64)) * 3).astype(np.float32), "bf16")
    k = synthetic.round_to((rng.normal(size=(B, T, 64)) * 3).astype(np.float32), "bf16")
    v = synthetic.round_to(rng.normal(size=(B, T, 64)).astype(np.float32), "bf16")
    out = to_np(wb.attention(_bf16(q), _bf16(k), _bf16(v), H))
    assert rel_l2(out[0], oenc.attention(q[0].astype(np.float64), k[0], v[0], H)) < 1e-2


@pytest.mark.parametrize("growth", [3.0, 12.0])
def test_attention_maxima_growing_along_the_keys(wb, growth):
    # scores rise steadily along the sequence, so the running row maxima move at some (growth 3) or
    # every (growth 12) later key tile: the paths that move the maxima and rescale O after tile 0
    rng = np.random.default_rng(int(growth))
    B, T, H = 1, 1500, 2
    base = rng.normal(size=(1, 1, 64 * H))
    q = synthetic.round_to((base + 0.1 * rng.normal(size=(B, T, 64 * H))).astype(np.float32), "bf16")
    ramp = (growth * np.arange(T) / T)[None, :, None]
    k = synthetic.round_to((base * ramp + 0.3 * rng.normal(size=(B, T, 64 * H))).astype(np.float32), "bf16")
    v = synthetic.round_to(rng.normal(size=(B, T, 64 * H)).astype(np.float32), "bf16")
    out = to_np(wb.attention(_bf16(q), _bf16(k), _bf16(v), H))
    assert wb.check_device_error() == 0
    assert rel_l2(out[0], oenc.attention(q[0].astype(np.float64), k[0], v[0], H)) < 1e-2


def test_attention_single_key_returns_v(wb):
    # T = 1: the only weight is 1 and the row sum is 1, so every output equals v (bf16 -> f16 -> bf16 is exact)
    rng = np.random.default_rng(5)
    B, T, H = 3, 1, 4
    q, k, v = (synthetic.round_to(rng.normal(size=(B, T, 64 * H)).astype(np.float32), "bf16") for _ in range(3))
    out = to_np(wb.attention(_bf16(q), _bf16(k), _bf16(v), H))
    assert wb.check_device_error() == 0
    np.testing.assert_array_equal(out, v)


@pytest.mark.parametrize("T", [1000, 1500])
def test_attention_zero_queries_average_values(wb, T):
    # q = 0: every score is 0, so each output row is the mean of the value rows over the sequence
    # (keys past T masked); closed form, independent of the oracle
    rng = np.random.default_rng(T)
    B, H = 2, 2
    q = np.zeros((B, T, 64 * H), np.float32)
    k, v = (synthetic.round_to(rng.normal(size=(B, T, 64 * H)).astype(np.float32), "bf16") for _ in range(2))
    out = to_np(wb.attention(_bf16(q), _bf16(k), _bf16(v), H))
    assert wb.check_device_error() == 0
    mean = v.astype(np.float64).mean(axis=1, keepdims=True)
    err = np.abs(out - mean)
    assert np.all(err <= 2.0 ** -8 * np.abs(mean) + 1e-4), float(err.max())


def test_device_error_word_clear(wb):
    assert wb.check_device_error() == 0


def test_gelu_epilogue_within_the_erfc_approximation_bound(wb):
    # zero operands: the FC1 epilogue returns GELU(bias) for a sweep of 4096 bias values.
    # The epilogue evaluates erfc by Abramowitz & Stegun 7.1.26 (|erf error| <= 1.5e-7), so
    # |GELU error| <= |x| * 0.75e-7 before the result is rounded to bf16 (half an ulp).
    N = 4096
    x = np.concatenate([np.linspace(-8, 8, N - 8), [0.0, 1e-3, -1e-3, 5.5, -5.5, 30.0, -30.0, 2.0]])
    bias = x.astype(np.float32)
    a = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((N, 64), dtype=torch.bfloat16, device=DEV)
    got = to_np(wb.linear(a, w, bias=_f32(bias), gelu=True))
    assert np.all(got == got[0:1])                                   # every row identical
    g = got[0]
    exact = oenc.gelu(bias.astype(np.float64))
    half_ulp = np.where(g != 0, 2.0 ** (np.floor(np.log2(np.abs(np.where(g != 0, g, 1.0)))) - 8), 0.0)
    bound = half_ulp + 0.75e-7 * np.abs(bias) * 1.001 + 2.0 ** -21 * np.abs(exact) + 1e-30
    assert np.all(np.abs(g - exact) <= bound), float(np.max(np.abs(g - exact) - bound))
    # away from the tail the result is the correctly rounded bf16 value or its neighbour
    ref = synthetic.round_to(exact.astype(np.float32), "bf16").astype(np.float64)
    body = np.abs(bias) <= 3
    assert np.all(np.abs(g - ref)[body] <= 2 * half_ulp[body] + 1e-30)
