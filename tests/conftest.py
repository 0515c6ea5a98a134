import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built liboscar.so")
    config.addinivalue_line("markers", "slow: large CPU oracle case")


@pytest.fixture(scope="session")
def liboscar():
    """Build (if stale) and load liboscar.so; the tests then call the C ABI through the binding."""
    from bit_kv_cache_write_gb300 import build, oscar
    build.build()
    return oscar.lib()


@pytest.fixture(scope="session")
def cuda(liboscar):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but CUDA is not available")
    return torch.device("cuda:0")
