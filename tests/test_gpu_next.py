"""GPU parity for the rows after the encoder path: decoder cross-attention K/V of
the encoder output, fused residual + RMSNorm, the E5M2 codec, and the
aggressive_fp8 preset (every encoder site in E4M3) per layer."""
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


def test_cross_kv_matches_oracle(wb):
    dims = synthetic.TINY
    rng = np.random.default_rng(5)
    enc_out = synthetic.round_to(rng.normal(size=(2, 1500, dims.d_model)).astype(np.float32), "bf16")
    layers = synthetic.cross_kv_weights(dims, 77, n_layers=3)
    dev_layers = [(_bf16(np.concatenate([L["wk"], L["wv"]])),
                   torch.as_tensor(np.concatenate([np.zeros(dims.d_model, np.float32), L["bv"]])).to(DEV))
                  for L in layers]
    kv = to_np(wb.cross_kv(_bf16(enc_out), dims, dev_layers))
    assert kv.shape == (3, 3000, 2 * dims.d_model)
    d = dims.d_model
    for b in range(2):
        ref = oenc.cross_kv(enc_out[b], layers)
        for l in range(3):
            rows = slice(b * 1500, (b + 1) * 1500)
            assert rel_l2(kv[l, rows, :d], ref[l][0]) < 1e-2
            assert rel_l2(kv[l, rows, d:], ref[l][1]) < 1e-2


@pytest.mark.parametrize("d,rows", [(1280, 1501), (384, 64)])
def test_rmsnorm_matches_oracle(wb, d, rows):
    rng = np.random.default_rng(d + 1)
    x = synthetic.round_to(rng.normal(0.2, 1.5, size=(rows, d)).astype(np.float32), "bf16")
    r = synthetic.round_to(rng.normal(size=(rows, d)).astype(np.float32), "bf16")
    g = (1 + 0.1 * rng.normal(size=d)).astype(np.float32)
    y, tot = wb.rmsnorm(_bf16(x), torch.as_tensor(g).to(DEV), residual=_bf16(r), return_total=True)
    assert rel_l2(to_np(y), oenc.rms_norm(x.astype(np.float64) + r, g)) < 4e-3
    y2 = wb.rmsnorm(_bf16(x), torch.as_tensor(g).to(DEV))
    assert rel_l2(to_np(y2), oenc.rms_norm(x.astype(np.float64), g)) < 4e-3


@pytest.mark.parametrize("n", [1000, 1280 * 1500 + 3])
def test_e5m2_bit_exact_vs_oracle_codec(wb, n):
    x = synthetic.round_to((np.random.default_rng(n).normal(size=n) * 5.0).astype(np.float32), "bf16")
    q, s = wb.quantize_e5m2(_bf16(x))
    q_ref, s_ref = ofp8.quantize_e5m2(x)
    assert s.item() == float(s_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    y = to_np(wb.dequantize_e5m2(q, s))
    ref = synthetic.round_to((ofp8.e5m2_decode(q_ref) * np.float64(s_ref)).astype(np.float32), "bf16")
    np.testing.assert_array_equal(y, ref)


def test_aggressive_fp8_tiny_and_large_layers(wb):
    sites = ("qkv", "out", "ffn")
    # tiny: one layer from the oracle's own input
    dims = synthetic.TINY
    w = synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32")
    _, enc = wb.upload_weights(w)
    enc.quantize()
    x0 = oenc.conv_stem(np.random.default_rng(3).uniform(-1.5, 1.5, (dims.n_mels, 3000)), w)
    x0d = _bf16(x0[None])
    out = to_np(wb.encoder_forward(x0d, dims, enc, precision=wb.PRESET_AGGRESSIVE_FP8, final_ln=False))[0]
    assert rel_l2(out, oenc.encoder(to_np(x0d)[0], w, dims.n_heads, final_ln=False, fp8_sites=sites)) < 6e-2
    # large-v3: the first four layers, each from the oracle's own input
    dims = synthetic.LARGE_V3
    w = synthetic.encoder_weights(dims, synthetic.SEED_LARGE_B1, "bf16", n_layers=4)
    w["ln_post_g"], w["ln_post_b"] = np.ones(dims.d_model, np.float32), np.zeros(dims.d_model, np.float32)
    _, enc = wb.upload_weights(w)
    enc.quantize()
    dims4 = synthetic.Dims(dims.n_mels, dims.d_model, dims.n_heads, 4, dims.d_ffn)
    h = oenc.conv_stem(np.random.default_rng(4).uniform(-1.5, 1.5, (dims.n_mels, 3000)), w)
    for layer in range(4):
        nxt = oenc.encoder_layer(h, w["layers"][layer], dims.n_heads, sites)
        got = to_np(wb.encoder_forward(_bf16(h[None]), dims4, enc, precision=wb.PRESET_AGGRESSIVE_FP8,
                                       layer_begin=layer, layer_end=layer + 1, final_ln=False))[0]
        assert rel_l2(got, nxt) < 6e-2, layer
        h = nxt
