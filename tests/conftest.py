import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


def pytest_collection_modifyitems(config, items):
    # GPU tests are never silently skipped on a GPU machine: a missing GPU or library there
    # is a failure. Here (no GPU) they are simply deselected with -m "not gpu".
    pass


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()
