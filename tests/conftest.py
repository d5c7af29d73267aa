import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: statistical oracle pins at full trial counts (minutes); "
                                       "run only when selected with -m slow")


def pytest_collection_modifyitems(config, items):
    # the full-power statistical pins run only when the marker expression
    # asks for them, so the default CPU suite stays within a few minutes
    if "slow" in (config.getoption("-m") or ""):
        return
    skip = pytest.mark.skip(reason="full-power statistical pin: select with -m slow")
    for item in items:
        if "slow" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def cuda_device():
    # GPU tests run only where a GPU is expected: a missing device is a
    # failure, not a skip, so that a broken box cannot pass silently.
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu but no CUDA device is visible")
    return torch.device("cuda:0")
