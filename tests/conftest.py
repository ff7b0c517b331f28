import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU oracle checks")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gdn():
    """The CUDA library binding; GPU tests fail loudly if it cannot be loaded."""
    if not cuda_available():
        pytest.skip("no CUDA device")
    from speculative_decode_gated_gdn_gb300 import lib
    return lib.load()
