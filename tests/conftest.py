import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-side preparation")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_matvec_gb300 import api
    return api
