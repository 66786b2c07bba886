import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


@pytest.fixture(scope="session")
def cuda_device():
    """The CUDA device for GPU tests; skips only when the machine has no GPU at all."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device on this machine")
    return torch.device("cuda:0")
