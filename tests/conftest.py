import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built library")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (compiled on first use if missing)."""
    from paged_kv_cache_317_gb300 import _build
    _build.build(quiet=True)
    from paged_kv_cache_317_gb300 import binding
    return binding.load_library()
