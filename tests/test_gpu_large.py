"""Full-size parity for Whisper large-v3 (GPU, through the C ABI).

  * batch 1 (seed 1000): every one of the 32 layers from the oracle's own
    input (relative L2 <= 1e-2 per layer) and the whole chain after the final
    LayerNorm (<= 3e-2), log-mel <= 1e-3 max abs, eagerly and replayed from a
    CUDA graph;
  * batch 32 (seeds 2000..2031): the last chunk against the oracle, and every
    chunk bitwise equal to the same chunk run alone (no cross-chunk coupling
    in bf16, a property that holds at any size);
  * mixed_fp8 at batch 32: every layer of the last chunk within 6e-2 of the
    oracle of the same pipeline (E4M3 operands at the qkv and ffn sites), the
    final output within a regression bound, chunks bitwise independent of
    their batch peers;
  * long-form 45 min (43.2 M samples, 108 windows at a 25 s stride, 3 batches
    of 36): log-mel of sampled windows <= 1e-3, the final zero-filled window
    through the whole encoder <= 3e-2.
The oracle runs one chunk at a time in float64 (about 45 s per chunk)."""
import dataclasses
import functools

import numpy as np
import pytest
import torch

from conftest import rel_l2, to_np
from oracle import encoder as oenc
from oracle import fp8 as ofp8
from oracle import frontend as ofe
import synthetic

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"
DIMS = synthetic.LARGE_V3


@functools.lru_cache(maxsize=2)
def host_weights(seed):
    return synthetic.encoder_weights(DIMS, seed, "bf16")


@functools.lru_cache(maxsize=2)
def device_weights(wb, seed):
    return wb.upload_weights(host_weights(seed))


@functools.lru_cache(maxsize=6)
def oracle_chain(seed, chunk_key, fp8=False):
    """(log-mel, stem output, residual after every layer, final output) for one chunk."""
    x = _chunk(chunk_key)
    w = host_weights(seed)
    mel = ofe.log_mel(x, DIMS.n_mels)
    x0 = oenc.conv_stem(mel, w)
    cap = []
    out = oenc.encoder(x0, w, DIMS.n_heads, capture=cap, fp8_sites=oenc.MIXED_FP8 if fp8 else ())
    return mel, x0, cap, out


@functools.lru_cache(maxsize=1)
def long_audio():
    return synthetic.long_audio(synthetic.SEED_LONGFORM)


def _chunk(key):
    kind, i = key
    if kind == "tone":
        return synthetic.tone_chunk(i)
    return ofe.chunk_audio(long_audio())[i]


def _dev(a):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def test_large_v3_batch1_per_layer_and_final(wb):
    seed = synthetic.SEED_LARGE_B1
    stem, enc = device_weights(wb, seed)
    mel_ref, x0_ref, cap, out_ref = oracle_chain(seed, ("tone", seed))
    audio = synthetic.tone_chunk(seed)
    pipe = wb.Pipeline(DIMS, stem, enc, batch=1)
    out = to_np(pipe(_dev(audio)))[0]
    assert wb.check_device_error() == 0
    assert np.abs(to_np(pipe.mel)[0] - mel_ref).max() <= 1e-3
    assert rel_l2(to_np(pipe.x0)[0], x0_ref) < 1e-2
    assert rel_l2(out, out_ref) < 3e-2
    worst = 0.0
    for layer in range(DIMS.n_layers):
        h_in = x0_ref if layer == 0 else cap[layer - 1]
        x = _dev(h_in[None]).to(torch.bfloat16)
        h = to_np(wb.encoder_forward(x, DIMS, enc, layer_begin=layer, layer_end=layer + 1, final_ln=False))[0]
        err = rel_l2(h, cap[layer])
        worst = max(worst, err)
        assert err < 1e-2, (layer, err)
    print(f"worst per-layer relative L2 {worst:.2e}")
    # the LayerNorm-kernel path (no folds) on the first and last layers
    enc_plain = wb.EncoderWeights([dataclasses.replace(L, ln_fold={}) for L in enc.layers], enc.ln_post_g,
                                  enc.ln_post_b)
    for layer in (0, DIMS.n_layers - 1):
        h_in = x0_ref if layer == 0 else cap[layer - 1]
        x = _dev(h_in[None]).to(torch.bfloat16)
        h = to_np(wb.encoder_forward(x, DIMS, enc_plain, layer_begin=layer, layer_end=layer + 1, final_ln=False))[0]
        assert rel_l2(h, cap[layer]) < 1e-2, layer


def test_large_v3_batch1_graph_replay_matches_oracle(wb):
    # the whole forward captured in a CUDA graph and replayed, against the float64 oracle
    seed = synthetic.SEED_LARGE_B1
    stem, enc = device_weights(wb, seed)
    mel_ref, _, _, out_ref = oracle_chain(seed, ("tone", seed))
    buf = _dev(synthetic.tone_chunk(seed))
    pipe = wb.Pipeline(DIMS, stem, enc, batch=1)
    graph = pipe.capture(buf)
    pipe.out.zero_()
    pipe.mel.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert wb.check_device_error() == 0
    assert np.abs(to_np(pipe.mel)[0] - mel_ref).max() <= 1e-3
    assert rel_l2(to_np(pipe.out)[0], out_ref) < 3e-2


@pytest.fixture(scope="module")
def batch32(wb):
    seed = synthetic.SEED_LARGE_B32
    stem, enc = device_weights(wb, seed)
    audio = synthetic.tone_batch(seed, 32)
    pipe = wb.Pipeline(DIMS, stem, enc, batch=32)
    out = pipe(_dev(audio.reshape(-1))).clone()
    mel = pipe.mel.clone()
    assert wb.check_device_error() == 0
    return stem, enc, audio, out, mel


def test_large_v3_batch32_last_chunk_matches_oracle(wb, batch32):
    _, _, audio, out, mel = batch32
    seed = synthetic.SEED_LARGE_B32
    mel_ref, _, _, out_ref = oracle_chain(seed, ("tone", seed + 31))
    assert np.abs(to_np(mel[31]) - mel_ref).max() <= 1e-3
    assert rel_l2(to_np(out[31]), out_ref) < 3e-2


def test_large_v3_batch32_chunks_independent_of_batch(wb, batch32):
    stem, enc, audio, out, _ = batch32
    pipe1 = wb.Pipeline(DIMS, stem, enc, batch=1)
    for b in range(32):
        one = pipe1(_dev(audio[b]))
        assert torch.equal(one[0], out[b]), b


def test_large_v3_batch32_mixed_fp8(wb, batch32):
    # E4M3 at the qkv and ffn sites, one activation scale per chunk.  Gate: every layer, fed the
    # oracle's own input, within 6e-2 of the oracle of the same pipeline.  End to end the E4M3
    # rounding decisions of two correct implementations diverge over 32 layers (bf16 storage
    # rounding moves values across E4M3 midpoints), so the final output is held to a looser
    # regression bound and reported.  Chunks are bitwise independent of their batch peers.
    stem, enc, audio, out_bf16, _ = batch32
    seed = synthetic.SEED_LARGE_B32
    pipe = wb.Pipeline(DIMS, stem, enc, batch=32, precision=wb.PRESET_MIXED_FP8)
    out = pipe(_dev(audio.reshape(-1))).clone()
    assert wb.check_device_error() == 0
    _, x0_8, cap8, ref8 = oracle_chain(seed, ("tone", seed + 31), fp8=True)
    worst = 0.0
    for layer in range(DIMS.n_layers):
        h_in = x0_8 if layer == 0 else cap8[layer - 1]
        x = _dev(h_in[None]).to(torch.bfloat16)
        h = to_np(wb.encoder_forward(x, DIMS, enc, precision=wb.PRESET_MIXED_FP8, layer_begin=layer,
                                     layer_end=layer + 1, final_ln=False))[0]
        err = rel_l2(h, cap8[layer])
        worst = max(worst, err)
        assert err < 6e-2, (layer, err)
    e2e8 = rel_l2(to_np(out[31]), ref8)
    _, _, _, ref = oracle_chain(seed, ("tone", seed + 31))
    e2e = rel_l2(to_np(out[31]), ref)
    print(f"mixed_fp8: worst per-layer relative L2 {worst:.3e}; final vs the E4M3 oracle {e2e8:.3e}, "
          f"vs the unquantised oracle {e2e:.3e}")
    # measured 6.45e-2 and 8.10e-2 on the code this bound was set on; a regression of more than
    # about 10 % fails
    assert e2e8 < 7e-2 and e2e < 9e-2
    # the float64 E4M3 oracle drifts from itself by this much when only its residual stream is stored
    # as bf16 between layers (tests/golden/fp8_drift.json, written from the oracle alone): a bf16
    # pipeline's distance from the E4M3 oracle is of that size, not a sign of a wrong decision
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "fp8_drift.json")) as fh:
        own = json.load(fh)["final_ln"]["e4m3_b_vs_e4m3"]
    print(f"mixed_fp8: E4M3 oracle with bf16 residual storage vs E4M3 oracle {own:.3e}")
    assert e2e8 < 1.2 * own
    pipe1 = wb.Pipeline(DIMS, stem, enc, batch=1, precision=wb.PRESET_MIXED_FP8)
    for b in (0, 17, 31):
        assert torch.equal(pipe1(_dev(audio[b]))[0], out[b]), b


def _site_codes(values, tol_flips, what):
    """Per-item E4M3 codes of the GPU and the oracle for one site, compared: the fraction that
    differs, and the size of each difference (one E4M3 step at most)."""
    q_gpu, q_ref, amax_gpu, amax_ref = values
    flips = q_gpu != q_ref
    frac = float(flips.mean())
    assert frac < tol_flips, (what, frac)
    dg, dr = ofp8.e4m3_decode(q_gpu[flips]), ofp8.e4m3_decode(q_ref[flips])
    assert np.all(np.abs(dg - dr) <= 2.0 ** -3 * np.maximum(np.abs(dg), np.abs(dr)) + 2.0 ** -9), what
    assert abs(amax_gpu - amax_ref) <= 2.0 ** -8 * amax_ref, what
    return frac


def test_large_v3_mixed_fp8_sites_from_identical_bf16_input(wb):
    # Where the GPU's E4M3 path departs from the E4M3 oracle, one site at a time.  Each side gets
    # the same bf16 input at the site (the GPU's own value of the previous step), so a code can
    # differ only where the site's value lies within one bf16 rounding of an E4M3 rounding
    # boundary (the GPU forms it in float32, the oracle in float64).  Measured: at most 4.3e-6 of
    # the codes (a handful per site), each one step, and the same per-chunk scale.  The FC1 GEMM + GELU fed the
    # same codes agrees with the oracle at bf16 accuracy.
    #
    # A whole layer fed the same bf16 input still ends about 2e-2 from the E4M3 oracle: the
    # residual after attention differs by bf16 rounding (relative delta ~ 2e-3), and a quantiser
    # with step u turns a perturbation delta << u into code flips on a fraction ~ delta / u of
    # the values, each of size u, i.e. a relative error ~ sqrt(delta * u) ~ sqrt(2e-3 * 0.09)
    # ~ 1.3e-2 at each of the two FFN sites.  That is a property of comparing a bf16 pipeline
    # with a float64 one across an E4M3 decision, not of either implementation.
    seed = synthetic.SEED_LARGE_B32
    _, enc = device_weights(wb, seed)
    enc.quantize()
    w = host_weights(seed)
    _, x0_8, cap8, _ = oracle_chain(seed, ("tone", seed + 31), fp8=True)
    T, D, H = 1500, DIMS.d_model, DIMS.n_heads
    f64 = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    report = []
    for layer in (0, 15, 31):
        L, Ld = w["layers"][layer], enc.layers[layer]
        x = ofp8.round_bf16(x0_8 if layer == 0 else cap8[layer - 1])
        xd = _dev(x).to(torch.bfloat16)
        # --- qkv site: LayerNorm 1 straight to codes
        q1, am1, _ = wb.layernorm_e4m3(xd, Ld.ln1_g, Ld.ln1_b, rows_per_item=T)
        c1, s1 = ofp8.quantize(ofp8.round_bf16(oenc.layer_norm(x, L["ln1_g"], L["ln1_b"])))
        f_qkv = _site_codes((to_np(q1).astype(np.uint8), c1, to_np(am1)[0], float(s1) * 448.0), 1e-4, "qkv")
        # the GPU's layer up to the residual after attention, from its own codes (building blocks)
        wq, sq = Ld.fp8["w_qkv"]
        qkv = wb.linear(q1, wq, bias=Ld.b_qkv, scale_a=am1 / 448.0, scale_w=sq)
        o = wb.attention(qkv[:, :D][None].contiguous(), qkv[:, D:2 * D][None].contiguous(),
                         qkv[:, 2 * D:][None].contiguous(), H)[0]
        h = wb.linear(o, Ld.w_out, bias=Ld.b_out, resid=xd)
        hx = to_np(h)
        # --- fc1 site: LayerNorm 2 of that residual straight to codes
        q2, am2, _ = wb.layernorm_e4m3(h, Ld.ln2_g, Ld.ln2_b, rows_per_item=T)
        c2, s2 = ofp8.quantize(ofp8.round_bf16(oenc.layer_norm(hx, L["ln2_g"], L["ln2_b"])))
        q2n = to_np(q2).astype(np.uint8)
        f_fc1 = _site_codes((q2n, c2, to_np(am2)[0], float(s2) * 448.0), 1e-4, "fc1")
        # --- fc2 site: GELU(FC1) of the GPU's fc1 codes, stored bf16, then per-chunk codes
        w1q, s1q = Ld.fp8["w_fc1"]
        g = wb.linear(q2, w1q, bias=Ld.b_fc1, scale_a=am2 / 448.0, scale_w=s1q, gelu=True)
        qg, sg = wb.quantize_fp8(g)
        a_deq = ofp8.e4m3_decode(q2n) * float(np.float32(to_np(am2)[0]) / np.float32(448.0))
        w_deq = ofp8.e4m3_decode(to_np(w1q).astype(np.uint8)) * float(to_np(s1q)[0])
        g_exact = oenc.gelu(a_deq @ w_deq.T + f64(L["b1"]))
        e_g = rel_l2(to_np(g), g_exact)
        assert e_g < 4e-3, (layer, e_g)                       # same codes in: bf16 accuracy out
        c3, s3 = ofp8.quantize(ofp8.round_bf16(g_exact))
        f_fc2 = _site_codes((to_np(qg).astype(np.uint8), c3, float(to_np(sg)[0]) * 448.0, float(s3) * 448.0),
                            1e-4, "fc2")
        # --- the whole layer from the identical bf16 input
        out = to_np(wb.encoder_forward(xd[None], DIMS, enc, precision=wb.PRESET_MIXED_FP8, layer_begin=layer,
                                       layer_end=layer + 1, final_ln=False))[0]
        ref = oenc.encoder(x, dict(w, layers=[L]), H, final_ln=False, fp8_sites=oenc.MIXED_FP8)
        err = rel_l2(out, ref)
        report.append((layer, f_qkv, f_fc1, f_fc2, e_g, err))
        assert err < 3e-2, (layer, err)                       # measured 2.2e-2 at layer 0
    for layer, a, b, c, eg, e in report:
        print(f"layer {layer}: code flips qkv {a:.2e} fc1 {b:.2e} fc2 {c:.2e}; FC1+GELU from the same codes "
              f"{eg:.2e}; layer from identical bf16 input {e:.2e}")
    assert wb.check_device_error() == 0


def test_long_form_45_min(wb):
    x = long_audio()
    n = ofe.n_chunks_for(len(x))
    assert n == 108
    seed = synthetic.SEED_LONGFORM
    stem, enc = device_weights(wb, seed)
    xd = _dev(x)
    pipe = wb.Pipeline(DIMS, stem, enc, batch=36)
    outs, mels = [], []
    for i in range(3):   # three batches of 36 windows through the same calls
        start = i * 36 * ofe.CHUNK_STRIDE
        outs.append(pipe(xd[start:], chunk_stride=ofe.CHUNK_STRIDE).clone())
        mels.append(pipe.mel.clone())
    assert wb.check_device_error() == 0
    chunks = ofe.chunk_audio(x)
    for c in (0, 35, 36, 71, 107):
        m = to_np(mels[c // 36][c % 36])
        assert np.abs(m - ofe.log_mel(chunks[c], DIMS.n_mels)).max() <= 1e-3, c
    _, _, _, out_ref = oracle_chain(seed, ("long", 107))
    assert rel_l2(to_np(outs[2][35]), out_ref) < 3e-2
