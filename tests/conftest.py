import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload on the GPU")


def _has_cuda() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_cuda():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """One line per workload: sequence decisions left out of the bit-exact comparison
    because a confidence lay within 1e-5 of gamma (or the floor compared confidences
    that close); they were checked for validity instead."""
    try:
        from gpu_util import EXCLUDED
    except Exception:
        return
    if not EXCLUDED:
        return
    terminalreporter.write_sep("-", "gamma-band exclusions (validity-checked, not bit-exact)")
    for key in sorted(EXCLUDED):
        n, total = EXCLUDED[key]
        terminalreporter.write_line(f"{key}: {n} of {total} sequence decisions excluded")
