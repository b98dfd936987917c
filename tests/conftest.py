import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


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


def pytest_terminal_summary(terminalreporter):
    """Worst achieved error of each parity rule in this run (GPU runs)."""
    try:
        from _helpers import ERRORS
    except ImportError:  # pragma: no cover
        return
    if not ERRORS:
        return
    terminalreporter.write_line("parity: worst achieved error / bound per rule")
    for name, (err, bound) in sorted(ERRORS.items()):
        terminalreporter.write_line(f"  {name:32s} {err:.3e} / {bound:.3e} = {err / bound:.3f}")
