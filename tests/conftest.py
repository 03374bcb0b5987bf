import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (builds it in-tree if needed; no GPU needed)."""
    from sparse_attention_step_gb300 import build, msa
    build.build()
    return msa.load()


def pytest_terminal_summary(terminalreporter):
    """Print the parity counts the GPU tests recorded (near-tie units at the
    selection boundary, summary elements that differ from the oracle's by one
    bf16 step), so they show even under -q."""
    try:
        from tests.parity import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    terminalreporter.write_line("parity counts:")
    for name, counts in REPORT:
        terminalreporter.write_line("  " + name + ": " + ", ".join(f"{k}={v}" for k, v in counts.items()))
