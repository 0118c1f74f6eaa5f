import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line(
        "markers", "slow: full-size workload; minutes of oracle time")


@pytest.fixture(scope="session")
def oracle():
    import oracle as oracle_pkg
    return oracle_pkg.load()


@pytest.fixture(scope="session")
def lib():
    """The product's C library, built in-tree if missing or stale."""
    from optimizer_step_resumable_gb300 import build as lib_build
    lib_build.build()
    import optimizer_step_resumable_gb300 as osr
    return osr.library()
