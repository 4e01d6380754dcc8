import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: longer CPU statistical tests")


def cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """Build (if needed) and load the CUDA library on a GPU host."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_70_gb300 import build as _b
    _b.build()
    import speculative_decoding_verification_70_gb300 as ssd
    ssd.load_library()
    return ssd
