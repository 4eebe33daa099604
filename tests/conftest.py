import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    """The compiled oracle; PF_ORACLE_SO names another build of it (the mutation test uses this)."""
    import oracle
    return oracle.load(os.environ.get("PF_ORACLE_SO") or None)
