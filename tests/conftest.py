import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libw4")


import pytest


def pytest_collection_modifyitems(config, items):
    # a per-test limit where the pytest-timeout plugin is installed (every device wait is bounded, so
    # a test that runs this long is stuck in a chain of expiring waits, not computing); the thread
    # method ends the process even while the main thread is blocked inside a CUDA call
    if not config.pluginmanager.hasplugin("timeout"):
        return
    for item in items:
        if item.get_closest_marker("timeout") is None:
            item.add_marker(pytest.mark.timeout(300, method="thread"))


@pytest.fixture(scope="session")
def libw4():
    """Builds libw4.so in-tree if it is missing or stale (nvcc cross-compiles without a GPU)."""
    from weight_only_bit_gb300 import build as _b
    _b.build()
    from weight_only_bit_gb300._lib import lib
    return lib()
