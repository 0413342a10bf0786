import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The built GPU library; a GPU test fails loudly when either is missing."""
    if not cuda_available():
        pytest.fail("gpu-marked test run without a CUDA device")
    import indirect_implicit_gemm_gb300 as g
    g.load()  # raises if libconvgb.so is absent
    return g
