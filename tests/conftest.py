import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a); runs the CUDA library")
    config.addinivalue_line("markers", "slow: large CPU case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library, loaded through the product binding (builds it if absent)."""
    from paged_mla_kv_cache_gb300 import build
    build.build_library()
    from paged_mla_kv_cache_gb300 import binding
    return binding.load_library()
