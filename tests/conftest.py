import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    """GPU tests are skipped, not failed, where no GPU is present, so that a
    plain `pytest tests/` on a CPU machine stays green."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Repeat the parity tests' count lines (code flips, stage errors) in the
    summary, where a run without -s still shows them."""
    parity = sys.modules.get("tests.parity")
    lines = getattr(parity, "REPORT", None) if parity else None
    if lines:
        terminalreporter.section("parity counts")
        for line in lines:
            terminalreporter.write_line(line)
