import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the libmsa kernels)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    # run the file that holds the standalone no-allocation entry point last
    items.sort(key=lambda it: ("test_zz" in it.nodeid,))


@pytest.fixture(scope="session")
def has_gpu():
    import torch
    return torch.cuda.is_available()
