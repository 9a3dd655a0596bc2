import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.lib()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Boundary-band counts of every oracle comparison of the run (see
    tests/band_report.py), printed even under -q."""
    try:
        import band_report
    except ImportError:
        return
    if not band_report.RECORDS:
        return
    terminalreporter.write_sep("-", "oracle parity: trials checked and boundary-band counts by kind")
    for line in band_report.table():
        terminalreporter.write_line(line)
