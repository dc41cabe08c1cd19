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


def pytest_terminal_summary(terminalreporter):
    # how often a clipped GPU step's clip coefficient came out one fp32 ulp
    # from the oracle's (checked then against the oracle's update with the
    # GPU's coefficient, bit for bit): per test and in total
    helpers = sys.modules.get("gpu_helpers")
    counts = getattr(helpers, "ULP_BRANCH", None)
    if not counts:
        return
    taken = sum(v[0] for v in counts.values())
    total = sum(v[1] for v in counts.values())
    terminalreporter.write_line("clipped GPU steps whose clip coefficient was one ulp off the oracle's: "
                                "%d of %d" % (taken, total))
    for name, (t, n) in sorted(counts.items()):
        if t:
            terminalreporter.write_line("  %s: %d of %d steps" % (name, t, n))
