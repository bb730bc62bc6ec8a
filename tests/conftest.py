import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


def cuda_ready() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def sdpa_lib():
    """The built sm_103a library (built here if missing); GPU tests only."""
    if not cuda_ready():
        pytest.skip("no CUDA device in this process")
    from scaled_dot_product_forward_gb300 import _build
    _build.build()
    import scaled_dot_product_forward_gb300 as sdpa
    sdpa.load_library()
    return sdpa
