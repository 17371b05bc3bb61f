import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


def pytest_terminal_summary(terminalreporter):
    from tests import _parity_log
    rows = _parity_log.lines()
    if rows:
        terminalreporter.write_sep("-", "parity: max-abs error vs the fp64 oracle")
        for ln in rows:
            terminalreporter.write_line(ln)
