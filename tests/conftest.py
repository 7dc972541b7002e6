import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints every float parity comparison (normwise and elementwise
    errors); MOE_PARITY_LOG=<path> also writes them as CSV."""
    from tests import parity_log
    lines = parity_log.summary_lines()
    if not lines:
        return
    terminalreporter.section("float parity (normwise / elementwise)")
    for line in lines:
        terminalreporter.write_line(line)
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        parity_log.write_csv(path)
