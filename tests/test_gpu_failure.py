"""Failure detection on the GPU without a fault (GPU).

Every wait inside libwb's kernels is bounded: when it runs out, the kernel
records ERR_TIMEOUT and the wait's site in the device error word and returns
normally.  The diagnostic entry point waits on an mbarrier that nothing
arrives on, so its wait always runs out; this checks that the timeout is
reported, that reading the word clears it, and that the context keeps
computing correct results afterwards."""
import ctypes
import time

import numpy as np
import pytest
import torch

from conftest import to_np
import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _small_linear(wb):
    a, w = synthetic.gemm_operands(11, 300, 256, 320, -1, 1)
    ref = a.astype(np.int64) @ w.astype(np.int64).T
    to_dev = lambda x: torch.as_tensor(np.asarray(x, np.float32)).to(DEV).to(torch.bfloat16)  # noqa: E731
    out = wb.linear(to_dev(a), to_dev(w))
    return to_np(out), ref.astype(np.float64)


def test_bounded_wait_reports_timeout_and_context_stays_usable(wb):
    from whisper_encoder_gb300 import _lib
    assert wb.check_device_error() == 0                  # nothing pending from earlier tests
    torch.cuda.synchronize()
    t0 = time.monotonic()
    wb.selftest_wait_timeout()
    raw = ctypes.c_uint32(0)
    st = _lib.load().wb_check_device_error(None, ctypes.byref(raw))
    elapsed = time.monotonic() - t0
    word = raw.value
    assert st == _lib.WB_ETIMEOUT
    assert word & 1, hex(word)                             # ERR_TIMEOUT
    assert (word >> 8) & 0xFF == _lib.WB_SELFTEST_WAIT_SITE, hex(word)
    assert 1.5 < elapsed < 60.0, elapsed                   # the wait's limit is about 2 s
    assert wb.check_device_error() == 0                  # reading the word cleared it

    got, ref = _small_linear(wb)                           # later launches run normally
    assert wb.check_device_error() == 0
    np.testing.assert_array_equal(got, ref)


def test_python_wrapper_returns_the_word_instead_of_raising(wb):
    from whisper_encoder_gb300 import _lib
    wb.selftest_wait_timeout(torch.cuda.current_stream())
    word = wb.check_device_error(torch.cuda.current_stream())
    assert word == 1 | (_lib.WB_SELFTEST_WAIT_SITE << 8)
    assert wb.check_device_error() == 0
