import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--exhaustive", action="store_true", default=False,
                     help="also run the exhaustive protocol searches (minutes of host work each)")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (seconds of host work)")
    config.addinivalue_line("markers", "exhaustive: a state-space search of minutes, run with --exhaustive")


def pytest_collection_modifyitems(config, items):
    if config.getoption("--exhaustive"):
        return
    skip = pytest.mark.skip(reason="exhaustive search: run with --exhaustive")
    for item in items:
        if "exhaustive" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def lib():
    """The CUDA library binding; GPU tests fail loudly if it is missing."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import tile_scheduling_gb300 as ts

    return ts


@pytest.fixture(scope="session")
def ts():
    """The binding for host-only calls (loads the built library; no GPU needed)."""
    import tile_scheduling_gb300 as ts

    return ts
