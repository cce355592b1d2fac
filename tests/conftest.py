import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Log how many bf16 outputs needed the half-ulp allowance of the output
    tolerance (expected to be about 0)."""
    parity = sys.modules.get("parity")
    if parity is None or not parity.ALLOWANCE["compared"]:
        return
    a = parity.ALLOWANCE
    terminalreporter.write_line(f"bf16 outputs within tolerance only by the half-ulp allowance: "
                                f"{a['used']} of {a['compared']}")
