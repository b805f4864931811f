"""Full-size parity for Whisper large-v3 (GPU, through the C ABI).

  * batch 1 (seed 1000): every one of the 32 layers from the oracle's own
    input (relative L2 <= 1e-2 per layer) and the whole chain after the final
    LayerNorm (<= 3e-2), log-mel <= 1e-3 max abs;
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
    assert e2e8 < 0.1 and e2e < 0.12
    pipe1 = wb.Pipeline(DIMS, stem, enc, batch=1, precision=wb.PRESET_MIXED_FP8)
    for b in (0, 17, 31):
        assert torch.equal(pipe1(_dev(audio[b]))[0], out[b]), b


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
