import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built extension")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, loaded through the product binding."""
    from token_dispatch_grouped_topk_gb300 import _lib
    return _lib.load()
