import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def dbuf_lib():
    """The CUDA library (libdbuf.so), built in-tree for sm_103a if stale."""
    from fsdp_infra_gb300 import build
    build.build()
    from fsdp_infra_gb300 import dbuf
    dbuf.library()
    return dbuf


_ORACLE_PLANS = {}


@pytest.fixture(scope="session")
def oracle_plans(oracle_lib):
    """Oracle plans of the five workloads, computed once per session."""
    from workloads import workload

    def get(key, gi):
        if (key, gi) not in _ORACLE_PLANS:
            w = workload(key)
            g = w.groups[gi]
            _ORACLE_PLANS[(key, gi)] = oracle_lib.plan_specs(g.tensors, w.m, w.local_units, w.align)
        return _ORACLE_PLANS[(key, gi)]
    return get
