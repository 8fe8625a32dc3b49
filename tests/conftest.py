import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libw4")
    # a per-test limit where the pytest-timeout plugin is installed (every device wait is bounded, so
    # a test that runs this long is stuck in a chain of expiring waits, not computing)
    if config.pluginmanager.hasplugin("timeout") and not getattr(config.option, "timeout", None):
        config.option.timeout = 600


import pytest


@pytest.fixture(scope="session")
def libw4():
    """Builds libw4.so in-tree if it is missing or stale (nvcc cross-compiles without a GPU)."""
    from weight_only_bit_gb300 import build as _b
    _b.build()
    from weight_only_bit_gb300._lib import lib
    return lib()
