import functools
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300 / sm_103a)")


@functools.lru_cache(maxsize=None)
def _workload(config, **kw):
    from sparse_selected_cell_gb300 import gen
    return gen.make(config, **kw)


@pytest.fixture(scope="session")
def workload():
    """workload(config_id, **overrides) -> cached generator Workload."""
    def get(config, **kw):
        return _workload(config, **kw)
    return get


@pytest.fixture(scope="session")
def oracle_lib():
    from oracle import oracle
    return oracle.load()
