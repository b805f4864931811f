"""CUDA-graph capture of the whole hot path (log-mel, stem, encoder): a replay
gives bitwise the eager result, and follows new contents of the input buffer."""
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
