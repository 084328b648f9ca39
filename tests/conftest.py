import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run on the GB300 box)")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (compiled by __graft_entry__.build() first)."""
    from context_attention_softmax_gb300 import _lib
    return _lib.load()
