import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libquoka.so")
    config.addinivalue_line("markers", "slow: full-size parity case (still part of the gpu suite)")


@pytest.fixture(scope="session")
def quoka():
    """The ctypes binding with libquoka.so built in-tree (nvcc cross-compiles without a GPU)."""
    from sparse_attention_chunked_gb300 import build as qbuild
    from sparse_attention_chunked_gb300 import quoka as qmod
    qbuild.build()
    qmod.load()
    return qmod
