import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--slow-oracle", action="store_true", default=False,
                     help="also run the comparisons whose oracle takes minutes")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow_oracle: the oracle side takes minutes; runs only "
                                       "with --slow-oracle")


def pytest_collection_modifyitems(config, items):
    if config.getoption("--slow-oracle"):
        return
    skip = pytest.mark.skip(reason="oracle takes minutes: run with --slow-oracle")
    for item in items:
        if "slow_oracle" in item.keywords:
            item.add_marker(skip)
