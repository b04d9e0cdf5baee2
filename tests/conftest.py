import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")
    # Test modules import the binding, which needs liblmc.so: (re)build it in
    # tree before collection when its sources are newer.
    _build_product()


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.lib()


def _build_product():
    import importlib.util
    path = os.path.join(ROOT, "state_cache_paging_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("lmc_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build_library()


@pytest.fixture(scope="session")
def lmc():
    """The product binding, built in-tree first if its sources changed."""
    _build_product()
    import state_cache_paging_gb300
    return state_cache_paging_gb300
