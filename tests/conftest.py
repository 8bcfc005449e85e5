import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built engine")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The worst error of each kind per test, next to its tolerance, so that
    the margins of a GPU run are on record in its log."""
    try:
        import harness
    except Exception:  # pragma: no cover
        return
    if not harness.MARGINS:
        return
    worst = {}
    for test, kind, value, tol in harness.MARGINS:
        key = (test, kind)
        if key not in worst or value > worst[key][0]:
            worst[key] = (value, tol)
    terminalreporter.section("parity margins (worst per test: value / tolerance)")
    for (test, kind), (value, tol) in sorted(worst.items()):
        terminalreporter.write_line(f"{value:.3e} / {tol:.0e}  {kind:<20} {test}")
