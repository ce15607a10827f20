import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def kvlib():
    """The built CUDA library; GPU tests skip when no device is present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_kv_cache_08_gb300 as kv
    kv.build()
    kv.lib()
    return kv
