import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Max-abs / mean-abs of the whole-output comparisons of the full-size
    workloads against the fp64 oracle (printed even with -q)."""
    try:
        from _helpers import PARITY_REPORT
    except Exception:
        return
    if not PARITY_REPORT:
        return
    terminalreporter.section("whole-output parity against the fp64 oracle")
    for what, n, mx, mean in PARITY_REPORT:
        terminalreporter.write_line(f"{what}: {n} elements, max-abs {mx:.3e}, mean-abs {mean:.3e}")
