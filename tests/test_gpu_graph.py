"""CUDA-graph capture of the whole hot path (log-mel, stem, encoder): a replay
gives bitwise the eager result, and follows new contents of the input buffer; the
pipelined host-to-host path (overlapped copies) gives the eager results."""
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


def test_run_host_overlapped_copies_match_eager(wb):
    # several batches from pinned host memory through Pipeline.run_host (double-buffered device
    # buffers, uploads and downloads on copy streams) give the eager results bitwise
    dims = synthetic.TINY
    stem, enc = wb.upload_weights(synthetic.encoder_weights(dims, synthetic.SEED_TINY, "f32"))
    B = 2
    pipe = wb.Pipeline(dims, stem, enc, batch=B)
    batches = [synthetic.tone_batch(700 + 10 * i, B).reshape(-1) for i in range(5)]
    host_in = [torch.from_numpy(a).pin_memory() for a in batches]
    host_out = [torch.empty(pipe.out.shape, dtype=torch.bfloat16).pin_memory() for _ in batches]
    pipe.run_host(host_in, host_out)
    torch.cuda.synchronize()
    assert wb.check_device_error() == 0
    for a, got in zip(batches, host_out):
        ref = pipe(torch.from_numpy(a).cuda()).cpu()
        assert torch.equal(got, ref)
