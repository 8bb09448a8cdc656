import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when run without a GPU: -m gpu is only run on a GPU machine.
    pass


@pytest.fixture(autouse=True)
def _output_guard_bands():
    """After every test: no kernel wrote into the sentinel bands around its output buffers."""
    yield
    if "gpu_util" in sys.modules:
        sys.modules["gpu_util"].check_guards()
