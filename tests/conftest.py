import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    import _report
    if not _report.PARITY:
        return
    terminalreporter.section("oracle parity (near ties: competing keys within 1e-4)")
    tot = dict(compared=0, exact=0, near_tie=0)
    for name, s in _report.PARITY:
        for k in tot:
            tot[k] += s[k]
        terminalreporter.write_line(
            f"{name}: compared {s['compared']}, exact {s['exact']}, near-tie {s['near_tie']}, "
            f"max score error {s['max_score_err']:.2e}")
    terminalreporter.write_line(
        f"all: compared {tot['compared']}, exact {tot['exact']}, near-tie {tot['near_tie']}")
