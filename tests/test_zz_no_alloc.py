"""wb_logmel_static, the log-mel entry point for callers that cannot allocate
device memory (it takes its scratch from a fixed array inside the library).

Called through the C ABI and compared with wb_logmel (caller workspace) on two
calls in a row: the second call uses fewer chunks and much quieter audio, so
per-chunk maxima left in the shared array by the first call would show up as
a wrong clamp.  This file sorts last so that a run stopping at its first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu
LOGMEL_TOL = 1e-3


def _static_call(wb, audio, n_chunks, n_mels, out):
    from whisper_encoder_gb300 import _lib
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.wb_logmel_static(ctypes.c_void_p(audio.data_ptr()), audio.numel(), 480000, n_chunks, n_mels,
                                ctypes.c_void_p(out.data_ptr()), stream)


def test_static_scratch_logmel_matches_workspace_logmel_twice(wb):
    from whisper_encoder_gb300 import _lib
    loud = torch.from_numpy(synthetic.tone_batch(4100, 2).reshape(-1)).cuda()
    quiet = torch.from_numpy((1e-3 * synthetic.tone_chunk(4200)).astype(np.float32)).cuda()
    for audio, n in ((loud, 2), (quiet, 1)):
        for n_mels in (128, 80):
            out = torch.full((n, n_mels, 3000), float("nan"), device="cuda")
            assert _static_call(wb, audio, n, n_mels, out) == _lib.WB_OK
            ref = wb.logmel(audio, n, n_mels)
            torch.cuda.synchronize()
            assert wb.check_device_error() == 0
            assert torch.isfinite(out).all()
            assert float((out - ref).abs().max()) <= LOGMEL_TOL


def test_static_scratch_rejects_more_chunks_than_it_holds(wb):
    from whisper_encoder_gb300 import _lib
    n = _lib.WB_LOGMEL_STATIC_MAX_CHUNKS + 1
    audio = torch.zeros(n * 480000, device="cuda")
    out = torch.full((n, 80, 3000), 7.0, device="cuda")
    assert _static_call(wb, audio, n, 80, out) == _lib.WB_EINVAL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())                     # nothing was launched
