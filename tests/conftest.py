import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Floating-point margins of the parity tests that ran: for each compared
    output, the plain max|gpu - oracle| / rms(oracle), and what is left of it
    beyond the per-element allowance (one bf16 ulp for bf16-stored outputs,
    the bf16 rounding of the dense baseline's dpre) against the tolerance."""
    try:
        from helpers import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.section("parity margins (max|err| / rms(ref))")
    tr.write_line(f"{'test':<72} {'output':<22} {'plain':>9} {'beyond allowance':>17} {'tol':>6}")
    for test, what, plain, beyond, tol in MARGINS:
        tr.write_line(f"{test[-72:]:<72} {what[:22]:<22} {plain:9.2e} {beyond:17.2e} {tol:6.0e}")
    worst = max(MARGINS, key=lambda m: m[3] / m[4])
    tr.write_line(f"largest share of the tolerance used: {worst[3] / worst[4]:.2f} ({worst[1]}, {worst[0]})")
