import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_terminal_summary(terminalreporter):
    """Print what the GPU parity tests recorded: per case, the elements compared
    and how many of them were beyond 1 ulp of the oracle (each one accepted only
    as cancellation, within the scale-relative bound)."""
    try:
        from tests import harness
    except Exception:
        return
    if harness.REPORT:
        terminalreporter.section("parity: elements beyond 1 ulp of the oracle")
        for line in harness.REPORT:
            terminalreporter.write_line(line)
