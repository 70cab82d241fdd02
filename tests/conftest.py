import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree for sm_103a; the test fails loudly if
    it cannot be built or loaded."""
    from selective_state_space_ssd_gb300 import binding
    return binding.load()
