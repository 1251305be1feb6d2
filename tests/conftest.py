import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")
    config.addinivalue_line("markers", "slow: full-size workloads (still part of the gpu suite)")


# Per-workload parity figures (max ulp, ulp histogram, max rstd error) that the
# full-size GPU tests collect, printed at the end of the run even without -s.
_PARITY_LINES: list = []


def pytest_sessionstart(session):
    _PARITY_LINES.clear()


def pytest_terminal_summary(terminalreporter):
    if _PARITY_LINES:
        terminalreporter.section("parity against the fp64 oracle (full size, every row)")
        for line in _PARITY_LINES:
            terminalreporter.write_line(line)


import pytest  # noqa: E402


@pytest.fixture
def parity_report():
    return _PARITY_LINES
