import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Achieved attention errors against the oracle, worst per test."""
    parity_util = sys.modules.get("parity_util")
    if parity_util is None or not parity_util.ACHIEVED:
        return
    worst = {}
    for label, dtype, a, r in parity_util.ACHIEVED:
        w = worst.get(label)
        worst[label] = (dtype, max(a, w[1]) if w else a, max(r, w[2]) if w else r,
                        (w[3] if w else 0) + 1)
    tr = terminalreporter
    tr.write_sep("-", "attention vs oracle: worst max-abs / relative error per test")
    for label, (dtype, a, r, n) in sorted(worst.items()):
        tr.write_line(f"{dtype:5s} max_abs {a:.3e}  rel {r:.3e}  ({n} checks)  {label}")
