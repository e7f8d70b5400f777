import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); runs the kernels through the C ABI")
    config.addinivalue_line("markers", "slow: long-running (full-size configs)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device here")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Element counts of the exhaustive full-size parity checks."""
    try:
        from tests import kvi_check
    except Exception:
        return
    if kvi_check.PARITY_LOG:
        terminalreporter.section("full-size parity: elements compared")
        for line in kvi_check.PARITY_LOG:
            terminalreporter.write_line(line)
