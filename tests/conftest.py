import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C ABI)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of host work)")


def golden_lines(name):
    """Non-comment, non-empty lines of a golden fixture, comments stripped."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line)
    return out


@pytest.fixture
def golden():
    return golden_lines


def pytest_terminal_summary(terminalreporter):
    """Near-tie counts of the code-parity tests (tests/tie_log.py)."""
    from tests import tie_log
    lines = tie_log.summary_lines()
    if lines:
        terminalreporter.section("near-tie counts (GPU codes vs oracle codes)")
        for line in lines:
            terminalreporter.write_line(line)
