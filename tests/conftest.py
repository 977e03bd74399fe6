import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Largest parity errors of the session (GPU tests), next to their tolerances."""
    try:
        from tests.helpers import RECORD, TOL
    except Exception:  # pragma: no cover
        return
    lines = []
    for dtype, book in RECORD.items():
        for key, (val, what) in sorted(book.items()):
            lines.append(f"{dtype:5s} {key:32s} {val:.3e}  (tolerance {TOL[dtype]:.0e})  at {what}")
    if lines:
        terminalreporter.write_sep("-", "largest parity errors against the fp64 oracle")
        for ln in lines:
            terminalreporter.write_line(ln)
