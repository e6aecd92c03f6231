import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
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


def pytest_terminal_summary(terminalreporter):
    """Achieved errors of the full-size parity checks (those that also assert
    the margin below the bars), as a table at the end of the run."""
    try:
        from tests import _util
    except Exception:  # pragma: no cover
        return
    if not _util.RECORD:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity margins (bars max-abs {_util.MAX_ABS:g} / mean-abs {_util.MEAN_ABS:g}; "
                      f"full-size checks held to {_util.MARGIN:.0%} of them)")
    for what, mx, mn, bmx, bmn in _util.RECORD:
        tr.write_line(f"{what}: max-abs {mx:.2e} ({mx / bmx:.1%} of bar), mean-abs {mn:.2e} ({mn / bmn:.1%} of bar)")
