import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size cases (minutes of host work)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle

    _oracle.build()
    return _oracle


def _cuda_ok():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def symar():
    """The CUDA library's Python binding, built in-tree; fails loudly when missing."""
    if not _cuda_ok():
        pytest.fail("GPU test collected on a host without CUDA")
    import symmetric_memory_allreduce_gb300 as sm

    sm.load()
    return sm
