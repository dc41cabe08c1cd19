"""pytest configuration: the ``gpu`` marker and shared fixtures."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libzero.so")
    # the suite imports the library: make sure it and the oracle are built
    # (incremental: a no-op when they are current)
    import __graft_entry__
    __graft_entry__.build()


def pytest_collection_modifyitems(config, items):
    # GPU tests run only where a GPU exists; elsewhere they are skipped, never faked.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
