import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def product_lib_path():
    """Builds (if stale) the C-ABI library and the oracle; returns the library path."""
    import __graft_entry__
    __graft_entry__.build()
    return os.path.join(ROOT, "deterministic_shot_all_gb300", "libarx.so")


@pytest.fixture(scope="session")
def arx(product_lib_path):
    """The Python binding of the C ABI (loads libarx.so)."""
    import deterministic_shot_all_gb300
    return deterministic_shot_all_gb300
