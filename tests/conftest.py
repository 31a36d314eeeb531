import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU and the built CUDA library")


def pytest_terminal_summary(terminalreporter):
    """The GEMM error margin per configuration, max and mean of |C - C_ref| / S
    over the compared elements (the bound is 2^-7), as the full-size parity
    tests recorded it."""
    gu = sys.modules.get("tests.gpu_util")
    margins = getattr(gu, "MARGINS", None) if gu is not None else None
    if not margins:
        return
    terminalreporter.write_sep("-", "GEMM error margin |C - C_ref| / S (bound 2^-7 = 7.81e-03)")
    for label, mx, mean, n in margins:
        terminalreporter.write_line(f"{label:44s} max {mx:.3e}  mean {mean:.3e}  ({n} elements)")
