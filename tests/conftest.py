import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    """The default oracle instance (compiled with gcc on first use)."""
    from oracle import oracle as _o
    path = os.environ.get("QMV_ORACLE_LIB")   # set only by the mutation tests
    return _o.Oracle(path) if path else _o.default()
