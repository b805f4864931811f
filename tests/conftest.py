import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libwb.so")
    config.addinivalue_line("markers", "slow: large oracle runs (seconds to minutes)")

import numpy as np  # noqa: E402
import pytest  # noqa: E402


@pytest.fixture(scope="session")
def wb():
    """The CUDA library, built for sm_103a; GPU tests fail (never skip) without it."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from whisper_encoder_gb300 import build
    build.build()
    import whisper_encoder_gb300 as w
    w.load()
    return w


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
