"""CUDA-graph capture of the whole hot path (log-mel, stem, encoder): a replay
gives bitwise the eager result, follows new contents of the input buffer and
matches the oracle; the host-to-host path through the C ABI (wb_encode_host,
with and without overlapped copies) gives the eager results and matches the
oracle."""
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision_name", ["PRESET_BF16", "PRESET_MIXED_FP8"])
def test_graph_replay_matches_eager(wb, precision_name):
    dims = synthetic.TINY
    stem, enc = wb.upload_weights(synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32"))
    precision = getattr(wb, precision_name)
    pipe = wb.Pipeline(dims, stem, enc, batch=2, precision=precision)
    a = torch.from_numpy(synthetic.tone_batch(300, 2).reshape(-1)).cuda()
    b = torch.from_numpy(synthetic.tone_batch(400, 2).reshape(-1)).cuda()
    buf = a.clone()
    graph = pipe.capture(buf)
    eager_a = pipe(a).clone()
    eager_b = pipe(b).clone()
    buf.copy_(a)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(pipe.out, eager_a)
    buf.copy_(b)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(pipe.out, eager_b)
    assert wb.check_device_error() == 0


@pytest.mark.parametrize("overlap", [True, False])
def test_run_host_overlapped_copies_match_eager(wb, overlap):
    # several batches from pinned host memory through wb_encode_host (double-buffered device
    # buffers, uploads and downloads on copy streams; or everything in order on one stream) give
    # the eager results bitwise
    dims = synthetic.TINY
    stem, enc = wb.upload_weights(synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32"))
    B = 2
    pipe = wb.Pipeline(dims, stem, enc, batch=B)
    batches = [synthetic.tone_batch(700 + 10 * i, B).reshape(-1) for i in range(5)]
    host_in = [torch.from_numpy(a).pin_memory() for a in batches]
    host_out = [torch.empty(pipe.out.shape, dtype=torch.bfloat16).pin_memory() for _ in batches]
    pipe.run_host(host_in, host_out, overlap=overlap)
    torch.cuda.synchronize()
    assert wb.check_device_error() == 0
    for a, got in zip(batches, host_out):
        ref = pipe(torch.from_numpy(a).cuda()).cpu()
        assert torch.equal(got, ref)


def test_graph_replay_matches_oracle_tiny(wb):
    # the replayed graph against the float64 oracle itself (log-mel <= 1e-3 max abs, output after
    # the final LayerNorm <= 3e-2; mixed_fp8 <= 6e-2 from the oracle with E4M3 qkv / ffn sites)
    import numpy as np
    from conftest import rel_l2, to_np
    from oracle import encoder as oenc
    from oracle import frontend as ofe
    dims = synthetic.TINY
    w = synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32")
    stem, enc = wb.upload_weights(w)
    audio = synthetic.tone_batch(500, 2)
    buf = torch.from_numpy(audio.reshape(-1)).cuda()
    for precision, sites, tol in ((wb.PRESET_BF16, (), 3e-2), (wb.PRESET_MIXED_FP8, oenc.MIXED_FP8, 6e-2)):
        pipe = wb.Pipeline(dims, stem, enc, batch=2, precision=precision)
        graph = pipe.capture(buf)
        pipe.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert wb.check_device_error() == 0
        for b in range(2):
            mel_ref = ofe.log_mel(audio[b], dims.n_mels)
            assert np.abs(to_np(pipe.mel[b]) - mel_ref).max() <= 1e-3
            ref = oenc.encoder(oenc.conv_stem(mel_ref, w), w, dims.n_heads, fp8_sites=sites)
            assert rel_l2(to_np(pipe.out[b]), ref) < tol, (precision, b)


def test_encode_host_matches_oracle(wb):
    # the C-ABI host-buffer path against the float64 oracle (log-mel + stem + layer + final LN)
    import numpy as np
    from conftest import rel_l2
    from oracle import encoder as oenc
    from oracle import frontend as ofe
    dims = synthetic.TINY
    w = synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32")
    stem, enc = wb.upload_weights(w)
    pipe = wb.Pipeline(dims, stem, enc, batch=2)
    audio = [synthetic.tone_batch(900 + 10 * i, 2) for i in range(3)]
    host_in = [torch.from_numpy(a.reshape(-1)).pin_memory() for a in audio]
    host_out = [torch.empty(pipe.out.shape, dtype=torch.bfloat16).pin_memory() for _ in audio]
    pipe.run_host(host_in, host_out)
    torch.cuda.synchronize()
    assert wb.check_device_error() == 0
    for a, got in zip(audio, host_out):
        for b in range(2):
            ref = oenc.encoder(oenc.conv_stem(ofe.log_mel(a[b], dims.n_mels), w), w, dims.n_heads)
            assert rel_l2(got[b].float().numpy().astype(np.float64), ref) < 3e-2


def test_encode_host_mixed_fp8_and_25s_stride(wb):
    # wb_encode_host with the mixed_fp8 preset and overlapping 30 s windows at a 25 s stride (the
    # long-form layout): bitwise the eager calls on the same windows
    dims = synthetic.TINY
    stem, enc = wb.upload_weights(synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32"))
    B, stride = 2, 400000
    pipe = wb.Pipeline(dims, stem, enc, batch=B, precision=wb.PRESET_MIXED_FP8)
    n_samples = (B - 1) * stride + 480000 - 1234          # the last window runs past the end (zero fill)
    batches = [synthetic.long_audio(3100 + i, n_samples) for i in range(3)]
    host_in = [torch.from_numpy(a).pin_memory() for a in batches]
    host_out = [torch.empty(pipe.out.shape, dtype=torch.bfloat16).pin_memory() for _ in batches]
    pipe.run_host(host_in, host_out, chunk_stride=stride)
    torch.cuda.synchronize()
    assert wb.check_device_error() == 0
    for a, got in zip(batches, host_out):
        ref = pipe(torch.from_numpy(a).cuda(), chunk_stride=stride).cpu()
        assert torch.equal(got, ref)
