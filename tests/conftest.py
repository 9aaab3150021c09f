import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line(
        "markers", "first_gpu_run: a GPU test of code that has not yet passed on a GPU; "
        "collected after the others, so that a run stopping at its first failure has "
        "already run every established test")


def pytest_collection_modifyitems(config, items):
    # stable sort: the forward pass's parity tests first (the evidence every
    # other result builds on), then the rest in file order, then the tests
    # of code that has not yet passed on a GPU
    items.sort(key=lambda item: (item.get_closest_marker("first_gpu_run") is not None,
                                 os.path.basename(str(item.fspath)) != "test_parity_gpu.py"))
