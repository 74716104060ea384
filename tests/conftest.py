import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionfinish(session, exitstatus):
    """With GCL_PARITY_LOG=<path>, write every parity check's measured errors (global, worst
    unit, worst row ratio) and its bar to <path>, one tab-separated line each."""
    path = os.environ.get("GCL_PARITY_LOG")
    if not path:
        return
    try:
        import parity
    except ImportError:
        return
    with open(path, "w") as f:
        for name, eg, eu, er, tol in parity.RECORD:
            f.write(f"{name}\t{eg:.3e}\t{eu:.3e}\t{er:.3e}\t{tol:g}\n")
