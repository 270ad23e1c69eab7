import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running statistical test")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle as O
    O.build()
    return O


# Lines that tests record for the end-of-run summary (flag budget fractions).
_REPORT = []


@pytest.fixture(scope="session")
def report():
    """report(line): print `line` in the terminal summary, even under -q."""
    return _REPORT.append


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if _REPORT:
        terminalreporter.section("measured rates")
        for line in _REPORT:
            terminalreporter.write_line(line)
