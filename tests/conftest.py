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


@pytest.fixture(scope="session")
def pf():
    """The CUDA library, built in-tree for sm_103a; GPU tests fail (not skip) when it cannot load."""
    from paged_kv_decode_pf_gb300 import _build
    _build.build()
    import paged_kv_decode_pf_gb300 as pf_mod
    pf_mod.lib()
    return pf_mod


_WORKLOADS = {}


@pytest.fixture(scope="session")
def config_workload():
    """Named workloads, generated once per session."""
    from workloads import make_config

    def get(index):
        if index not in _WORKLOADS:
            _WORKLOADS[index] = make_config(index)
        return _WORKLOADS[index]
    return get
