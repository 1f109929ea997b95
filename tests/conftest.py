import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size case, minutes of CPU work")


def pytest_collection_modifyitems(config, items):
    # run the no-GPU suite quickly: nothing here needs a particular order
    pass


@pytest.fixture(scope="session")
def has_gpu():
    import torch
    return torch.cuda.is_available()
