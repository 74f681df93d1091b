import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The plain max |O_gpu - O_ref| of every forward comparison and the worst per-head
    relative gradient errors of the full-shape backward comparisons."""
    import foxtest

    if not foxtest.PARITY_LOG:
        return
    terminalreporter.section("parity against the oracle")
    for label, value, count in foxtest.PARITY_LOG:
        if isinstance(value, dict):
            body = " ".join(f"{k}={v:.2e}" for k, v in value.items())
            terminalreporter.write_line(f"{label}: {body} ({count} heads)")
        else:
            terminalreporter.write_line(f"{label}: max|dO| = {value:.3e} ({count} elements with |O_ref| >= 4)")
