"""Pins of the oracle's conv stem and encoder layers against closed forms,
brute force and torch's own float64 CPU modules (library special cases).  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import encoder as enc
oenc = enc
import synthetic

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_gelu_values():
    assert enc.gelu(0.0) == 0.0
    assert enc.gelu(1.0) == pytest.approx(0.8413447460685429, abs=1e-15)     # Phi(1)
    assert enc.gelu(-1.0) == pytest.approx(-0.15865525393145707, abs=1e-15)  # -(1 - Phi(1))
    assert enc.gelu(12.0) == pytest.approx(12.0, abs=1e-20)
    x = np.linspace(-6, 6, 1001)
    ref = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(enc.gelu(x), ref, atol=1e-15)


@pytest.mark.parametrize("d", [384, 1280])
def test_sinusoid_special_values(d):
    pe = enc.sinusoids(1500, d)
    h = d // 2
    t = np.arange(1500)
    assert np.all(pe[0, :h] == 0.0) and np.all(pe[0, h:] == 1.0)
    np.testing.assert_allclose(pe[:, 0], np.sin(t), atol=1e-12)
    np.testing.assert_allclose(pe[:, h], np.cos(t), atol=1e-12)
    np.testing.assert_allclose(pe[:, h - 1], np.sin(t / 10000.0), atol=1e-12)   # slowest: 1/10000
    np.testing.assert_allclose(pe[:, d - 1], np.cos(t / 10000.0), atol=1e-12)


@pytest.mark.parametrize("stride", [1, 2])
def test_conv1d_matches_torch_and_brute_force(stride):
    rng = np.random.default_rng(stride)
    x = rng.normal(size=(5, 11))
    w = rng.normal(size=(4, 5, 3))
    b = rng.normal(size=4)
    out = enc.conv1d_k3(x, w, b, stride)
    ref = torch.nn.functional.conv1d(torch.tensor(x)[None], torch.tensor(w), torch.tensor(b),
                                     stride=stride, padding=1)[0].numpy()
    np.testing.assert_allclose(out, ref, atol=1e-13)
    bf = np.zeros_like(out)
    for c in range(4):
        for t in range(out.shape[1]):
            s = b[c]
            for ci in range(5):
                for j in range(3):
                    i = stride * t + j - 1
                    if 0 <= i < 11:
                        s += w[c, ci, j] * x[ci, i]
            bf[c, t] = s
    np.testing.assert_allclose(out, bf, atol=1e-13)


def test_stem_identity_taps_reduce_to_gelu_and_even_frames():
    C = 8
    x = np.random.default_rng(0).normal(size=(C, 3000))
    w = {"conv1_w": np.zeros((C, C, 3)), "conv1_b": np.zeros(C),
         "conv2_w": np.zeros((C, C, 3)), "conv2_b": np.zeros(C)}
    w["conv1_w"][:, :, 1] = np.eye(C)
    w["conv2_w"][:, :, 1] = np.eye(C)
    x0 = enc.conv_stem(x, w)
    assert x0.shape == (1500, C)
    expect = enc.gelu(enc.gelu(x))[:, ::2].T + enc.sinusoids(1500, C)
    np.testing.assert_allclose(x0, expect, atol=1e-14)


def test_stem_matches_torch_modules():
    dims = synthetic.TINY
    w = synthetic.encoder_weights(dims, 5, "f32")
    mel = np.random.default_rng(2).uniform(-1.5, 1.5, size=(dims.n_mels, 3000))
    F = torch.nn.functional
    t = lambda a: torch.tensor(np.asarray(a, np.float64))  # noqa: E731
    y1 = F.gelu(F.conv1d(t(mel)[None], t(w["conv1_w"]), t(w["conv1_b"]), padding=1))
    y2 = F.gelu(F.conv1d(y1, t(w["conv2_w"]), t(w["conv2_b"]), stride=2, padding=1))[0].T.numpy()
    np.testing.assert_allclose(enc.conv_stem(mel, w), y2 + enc.sinusoids(1500, dims.d_model), atol=1e-12)


def test_layer_norm_moments_and_torch():
    eps = GOLDEN["layernorm_eps"]["value"]
    assert enc.LN_EPS == eps
    x = np.random.default_rng(3).normal(2.0, 3.0, size=(64, 1280))
    y = enc.layer_norm(x, np.ones(1280), np.zeros(1280))
    np.testing.assert_allclose(y.mean(1), 0.0, atol=1e-12)
    var = x.var(1)
    np.testing.assert_allclose(y.var(1), var / (var + eps), rtol=1e-12)
    g = np.random.default_rng(4).normal(size=1280)
    b = np.random.default_rng(5).normal(size=1280)
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (1280,), torch.tensor(g), torch.tensor(b), eps).numpy()
    np.testing.assert_allclose(enc.layer_norm(x, g, b), ref, atol=1e-12)


def test_softmax_rows_sum_to_one_and_shift_invariance():
    s = np.random.default_rng(6).normal(0, 30, size=(40, 1500))
    p = enc.softmax(s)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-13)
    assert (p >= 0).all()
    np.testing.assert_allclose(enc.softmax(s + 123.0), p, atol=1e-15)


def _brute_attention(q, k, v, H):
    T, d = q.shape
    hd = d // H
    out = np.zeros((T, d))
    for h in range(H):
        for i in range(T):
            sc = [sum(q[i, h * hd + e] * k[j, h * hd + e] for e in range(hd)) / math.sqrt(hd) for j in range(T)]
            m = max(sc)
            ex = [math.exp(s - m) for s in sc]
            z = sum(ex)
            for e in range(hd):
                out[i, h * hd + e] = sum(ex[j] * v[j, h * hd + e] for j in range(T)) / z
    return out


@pytest.mark.parametrize("T", [7, 13])
def test_attention_brute_force(T):
    rng = np.random.default_rng(T)
    q, k, v = (rng.normal(size=(T, 16)) for _ in range(3))
    np.testing.assert_allclose(enc.attention(q, k, v, 2), _brute_attention(q, k, v, 2), atol=1e-13)


def test_attention_matches_torch_sdpa_with_tail():
    T, H, hd = 130, 3, 64
    rng = np.random.default_rng(9)
    q, k, v = (rng.normal(size=(T, H * hd)) for _ in range(3))
    th = lambda a: torch.tensor(a).view(T, H, hd).transpose(0, 1)  # noqa: E731
    ref = torch.nn.functional.scaled_dot_product_attention(th(q), th(k), th(v)).transpose(0, 1).reshape(T, H * hd)
    np.testing.assert_allclose(enc.attention(q, k, v, H), ref.numpy(), atol=1e-12)


def test_attention_invariants():
    T, d = 50, 128
    rng = np.random.default_rng(10)
    q, v = rng.normal(size=(T, d)), rng.normal(size=(T, d))
    same = np.tile(rng.normal(size=(1, d)), (T, 1))
    np.testing.assert_allclose(enc.attention(q, same, v, 2), np.tile(v.mean(0), (T, 1)), atol=1e-13)
    k = rng.normal(size=(T, d)) * 0.01
    k[17] = q.sum(0) * 1000.0                   # one key dominates every score row
    out = enc.attention(np.abs(q) + 1.0, np.abs(k), v, 1)
    np.testing.assert_allclose(out, np.tile(v[17], (T, 1)), atol=1e-9)
    k = rng.normal(size=(T, d))
    np.testing.assert_allclose(enc.attention(q, k + rng.normal(size=(1, d)), v, 2),
                               enc.attention(q, k, v, 2), atol=1e-12)   # key bias is a no-op


def _torch_layer(L, d, H, F):
    layer = torch.nn.TransformerEncoderLayer(d, H, F, dropout=0.0, activation="gelu", batch_first=True,
                                             norm_first=True, dtype=torch.float64)
    t = lambda a: torch.tensor(np.asarray(a, np.float64))  # noqa: E731
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(torch.cat([t(L["wq"]), t(L["wk"]), t(L["wv"])]))
        layer.self_attn.in_proj_bias.copy_(torch.cat([t(L["bq"]), torch.zeros(d, dtype=torch.float64), t(L["bv"])]))
        layer.self_attn.out_proj.weight.copy_(t(L["wo"]))
        layer.self_attn.out_proj.bias.copy_(t(L["bo"]))
        layer.norm1.weight.copy_(t(L["ln1_g"])); layer.norm1.bias.copy_(t(L["ln1_b"]))
        layer.norm2.weight.copy_(t(L["ln2_g"])); layer.norm2.bias.copy_(t(L["ln2_b"]))
        layer.linear1.weight.copy_(t(L["w1"])); layer.linear1.bias.copy_(t(L["b1"]))
        layer.linear2.weight.copy_(t(L["w2"])); layer.linear2.bias.copy_(t(L["b2"]))
    return layer.eval()


def test_encoder_layer_matches_torch_transformer_layer():
    dims = synthetic.TINY
    w = synthetic.encoder_weights(dims, 21, "f32")
    L = w["layers"][0]
    h = np.random.default_rng(1).normal(size=(97, dims.d_model))
    ref = _torch_layer(L, dims.d_model, dims.n_heads, dims.d_ffn)(torch.tensor(h)[None])[0].detach().numpy()
    np.testing.assert_allclose(enc.encoder_layer(h, L, dims.n_heads), ref, atol=1e-11)


def test_encoder_runs_65_layernorms_for_large_v3(monkeypatch):
    facts = GOLDEN
    count = {"n": 0}
    orig = enc.layer_norm

    def counting(*a, **k):
        count["n"] += 1
        return orig(*a, **k)

    monkeypatch.setattr(enc, "layer_norm", counting)
    monkeypatch.setattr(enc, "attention", lambda q, k, v, H: q)       # shape-only stand-ins
    monkeypatch.setattr(enc, "gelu", lambda x: x)
    d = 8
    lay = {k: np.zeros(s) for k, s in [("ln1_g", d), ("ln1_b", d), ("bq", d), ("bv", d), ("bo", d), ("ln2_g", d),
                                        ("ln2_b", d), ("b1", d), ("b2", d)]}
    for k in ("wq", "wk", "wv", "wo", "w1", "w2"):
        lay[k] = np.zeros((d, d))
    w = {"layers": [lay] * synthetic.LARGE_V3.n_layers, "ln_post_g": np.ones(d), "ln_post_b": np.zeros(d)}
    enc.encoder(np.zeros((3, d)), w, 1)
    assert count["n"] == 65
    assert count["n"] + facts["decoder_layernorms"]["value"] == facts["layernorms_in_model"]["value"]


def test_encoder_capture_and_layer_range():
    dims = synthetic.TINY
    w = synthetic.encoder_weights(dims, 3, "f32")
    w["layers"] = w["layers"] * 2
    x0 = np.random.default_rng(0).normal(size=(20, dims.d_model))
    cap = []
    out = enc.encoder(x0, w, dims.n_heads, capture=cap)
    assert len(cap) == 2
    h1 = enc.encoder(x0, w, dims.n_heads, 0, 1, final_ln=False)
    np.testing.assert_array_equal(h1, cap[0])
    np.testing.assert_array_equal(enc.encoder(h1, w, dims.n_heads, 1, 2), out)


def _grid_layer(rng, d, F, beta_on_grid=True):
    """A layer whose quantised operands all sit exactly on their per-tensor E4M3 grid."""
    from oracle import fp8 as q8
    grid = q8.e4m3_decode(np.arange(0x00, 0x7F))                 # non-negative E4M3 values
    pick = lambda shape, s: (rng.choice(grid[grid <= 448], size=shape) *        # noqa: E731
                             rng.choice([-1.0, 1.0], size=shape)) * s
    def with_amax(w):                                              # force amax == 448 * s exactly
        w = w.copy(); w.flat[0] = 448.0 * (2.0 ** -12); return w
    L = {"ln1_g": np.zeros(d), "ln2_g": np.zeros(d)}
    L["ln1_b"] = with_amax(pick(d, 2.0 ** -12)) if beta_on_grid else rng.normal(size=d) * 0.05
    L["ln2_b"] = with_amax(pick(d, 2.0 ** -12))
    for k in ("wq", "wk", "wv"):
        L[k] = pick((d, d), 2.0 ** -14)
    L["wq"].flat[0] = 448.0 * 2.0 ** -14                           # fused QKV amax on the grid
    L["wo"] = rng.normal(size=(d, d)) * 0.02
    L["bq"], L["bv"], L["bo"] = (rng.normal(size=d) * 0.02 for _ in range(3))
    L["w1"], L["b1"] = np.zeros((F, d)), np.zeros(F)               # GELU(0) = 0: FC2 input exact
    L["w2"], L["b2"] = pick((d, F), 2.0 ** -14), rng.normal(size=d) * 0.02
    return L


def test_fp8_sites_are_exact_when_operands_sit_on_the_e4m3_grid():
    rng = np.random.default_rng(8)
    d, F, H = 128, 256, 2
    L = _grid_layer(rng, d, F)
    h = rng.normal(size=(40, d))
    ref = oenc.encoder_layer(h, L, H)
    np.testing.assert_allclose(oenc.encoder_layer(h, L, H, oenc.MIXED_FP8), ref, atol=1e-12)
    np.testing.assert_allclose(oenc.encoder_layer(h, L, H, ("qkv", "out", "ffn")) - ref,
                               oenc.encoder_layer(h, L, H, ("out",)) - ref, atol=1e-12)


def test_fp8_sites_quantise_off_grid_operands():
    rng = np.random.default_rng(9)
    d, F, H = 128, 256, 2
    L = _grid_layer(rng, d, F, beta_on_grid=False)
    h = rng.normal(size=(40, d))
    ref = oenc.encoder_layer(h, L, H)
    diff = np.abs(oenc.encoder_layer(h, L, H, ("qkv",)) - ref).max()
    assert 1e-6 < diff < 0.1 * np.abs(ref).max()                   # the QKV input was rounded
    assert np.abs(oenc.encoder_layer(h, L, H, ("ffn",)) - ref).max() < 1e-12   # FC1 input on grid, FC2 input 0


def test_rms_norm_matches_torch_and_unit_rms():
    x = np.random.default_rng(12).normal(0.5, 2.0, size=(33, 1280))
    g = np.random.default_rng(13).normal(size=1280)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (1280,), torch.tensor(g), 1e-5).numpy()
    np.testing.assert_allclose(enc.rms_norm(x, g), ref, atol=1e-12)
    y = enc.rms_norm(x, np.ones(1280))
    ms = (x * x).mean(1)
    np.testing.assert_allclose((y * y).mean(1), ms / (ms + 1e-5), rtol=1e-12)


def test_cross_kv_drives_torch_cross_attention():
    # the oracle's K / V, used as key and value of a softmax attention, reproduce torch's
    # MultiheadAttention(query, memory, memory) with the same projection weights
    d, H, T, Tq = 64, 2, 40, 7
    rng = np.random.default_rng(14)
    L = {"wk": rng.normal(size=(d, d)) * 0.1, "wv": rng.normal(size=(d, d)) * 0.1, "bv": rng.normal(size=d) * 0.1}
    wq, bq = rng.normal(size=(d, d)) * 0.1, rng.normal(size=d) * 0.1
    wo, bo = np.eye(d), np.zeros(d)
    mem = rng.normal(size=(T, d))
    query = rng.normal(size=(Tq, d))
    (k, v), = enc.cross_kv(mem, [L])
    q = query @ wq.T + bq
    hd = d // H
    ours = np.concatenate([enc.softmax(q[:, h * hd:(h + 1) * hd] @ k[:, h * hd:(h + 1) * hd].T / math.sqrt(hd))
                           @ v[:, h * hd:(h + 1) * hd] for h in range(H)], axis=1) @ wo.T + bo
    mha = torch.nn.MultiheadAttention(d, H, bias=True, batch_first=True, dtype=torch.float64)
    with torch.no_grad():
        mha.in_proj_weight.copy_(torch.tensor(np.concatenate([wq, L["wk"], L["wv"]])))
        mha.in_proj_bias.copy_(torch.tensor(np.concatenate([bq, np.zeros(d), L["bv"]])))
        mha.out_proj.weight.copy_(torch.tensor(wo)); mha.out_proj.bias.copy_(torch.tensor(bo))
    ref = mha(torch.tensor(query)[None], torch.tensor(mem)[None], torch.tensor(mem)[None])[0][0].detach().numpy()
    np.testing.assert_allclose(ours, ref, atol=1e-12)
