import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 and the built CUDA library")
    config.addinivalue_line(
        "markers", "slow: full-size workloads (minutes on a GB300)")


def pytest_collection_modifyitems(config, items):
    # a GPU test without a GPU is an error, not a skip: the product path has
    # no CPU fallback, so "-m gpu" on a CPU-only box must fail loudly.
    pass
