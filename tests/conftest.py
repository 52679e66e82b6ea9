import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built liblce.so")
    config.addinivalue_line("markers", "slow: full-size parity cases (minutes of float64 CPU work)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The ctypes binding with its library loaded; fails loudly when the
    CUDA library has not been built."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    import linear_cross_entropy_lce_gb300 as lce

    lce.load_library()
    return lce
