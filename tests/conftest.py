import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103) and the built C-ABI library")


@pytest.fixture(scope="session")
def lib():
    """The loaded C-ABI library (built in-tree by ``__graft_entry__.build``)."""
    from sequence_exact_attention_gb300 import binding
    return binding.load()
