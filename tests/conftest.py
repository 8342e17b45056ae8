import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (parity tests through the C ABI)")
    config.addinivalue_line("markers", "slow: full-size workload")


def pytest_terminal_summary(terminalreporter):
    """Print the worst err / bound ratio of each attention parity check, so
    the margin under the tolerance is visible in the run's output."""
    h = sys.modules.get("harness")
    worst = getattr(h, "WORST_RATIO", None) if h is not None else None
    if not worst:
        return
    terminalreporter.write_sep("-", "attention parity: worst |err| / bound per check")
    for name in sorted(worst):
        terminalreporter.write_line("%-60s %.3f" % (name, worst[name]))
