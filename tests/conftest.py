import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


# GPU test files that run after all the others (in this order): the backward pass is
# checked once the forward's tests have all run, and the allocation-free entry point last
# of all, so that a run stopping at its first failure has run every other test by then.
LAST = ("test_gpu_backward.py", "test_zz_no_alloc.py")


def pytest_collection_modifyitems(config, items):
    rank = {name: i + 1 for i, name in enumerate(LAST)}
    items.sort(key=lambda it: rank.get(os.path.basename(it.nodeid.split("::")[0]), 0))  # stable
    # Run GPU tests only where a GPU exists; on a CPU-only machine they are skipped
    # (the CPU suite is selected with -m "not gpu" anyway).
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
