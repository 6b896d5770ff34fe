import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large CPU case")


@pytest.fixture(scope="session")
def cpdr_lib():
    """Build (if stale) and load libcpdr.so; no GPU needed to load it."""
    from context_merge_gb300 import build as _build
    _build.build()
    from context_merge_gb300 import cpdr
    return cpdr.load()


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False
