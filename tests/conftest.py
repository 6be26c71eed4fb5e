import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libbevpool.so")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


@pytest.fixture(scope="session")
def wl_cache():
    """Workloads are deterministic; generate each one once per session."""
    from depth_weighted_scatter_gb300 import workloads

    cache = {}

    def get(name):
        if name not in cache:
            cache[name] = workloads.make(name)
        return cache[name]

    return get
