import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300 / sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


def pytest_terminal_summary(terminalreporter):
    """Steps compared, near-tie steps and the largest logit error of every parity run."""
    try:
        from parity import REPORTS
    except ImportError:
        return
    if not REPORTS:
        return
    terminalreporter.section("parity against the oracle")
    for name, steps, ties, err in REPORTS:
        terminalreporter.write_line(f"{name}: {steps} steps, {ties} near-tie steps, max |dz| (/std for bf16) {err:.4g}")
