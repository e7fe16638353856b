import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    try:
        from _parity import ALLOWANCE_LOG
    except Exception:  # pragma: no cover
        return
    if not ALLOWANCE_LOG:
        return
    tr = terminalreporter
    tr.section("derived flip allowances (units with an allowance / units, max allowance / max|ref|)")
    for test, what, n, total, mx in ALLOWANCE_LOG:
        tr.write_line("%s  %-16s %5d / %-6d %.2e" % (test, what, n, total, mx))
