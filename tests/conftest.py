import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size oracle comparisons (minutes of CPU)")


@pytest.fixture(scope="session")
def tp():
    """The ctypes binding of the C-ABI library (built in-tree)."""
    from tensor_transformer_layer_03_b300 import tp as binding
    return binding
