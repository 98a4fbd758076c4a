import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_terminal_summary(terminalreporter):
    """Print the error figures of the whole-tensor parity comparisons, if any ran."""
    import parity

    if parity.REPORT:
        terminalreporter.write_sep("-", "parity errors against the fp64 oracle")
        for name, err in parity.REPORT:
            terminalreporter.write_line(f"{name}: {err}")
