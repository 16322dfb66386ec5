import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when no GPU is present: the product has
    # no CPU fallback.  Deselect them with -m "not gpu" on a machine without one.
    pass


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
