import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and libkvarn")


@pytest.fixture(scope="session")
def kv():
    """The libkvarn binding; GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_kv_cache_kvarn_gb300 as kv

    kv.load()  # raises if the shared library is missing: no fallback path exists
    return kv
