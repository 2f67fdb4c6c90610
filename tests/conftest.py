import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-batch parity counts (requests compared, near-tie decisions by kind)."""
    from tests._compare import REPORT
    if REPORT:
        terminalreporter.section("parity with the oracle")
        for ln in REPORT:
            terminalreporter.write_line(ln)
