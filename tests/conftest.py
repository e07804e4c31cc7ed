import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # The CUDA library is built in-tree (incrementally) before any test module imports the
    # binding; a failed build fails the session loudly.
    import __graft_entry__
    __graft_entry__.build()


def read_golden(name: str) -> list[str]:
    """Non-comment, non-empty lines of a golden fixture."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


@pytest.fixture
def golden():
    return read_golden


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst parity margins of the bf16-I/O comparisons that ran (GPU tests only)."""
    mod = sys.modules.get("_gpu")
    if mod is None or not getattr(mod, "MARGINS", None):
        return
    terminalreporter.section("parity margins (bf16 I/O; bound = 2e-2 RMS(ref) + 2^-8 |ref| if stored in bf16)")
    for line in mod.margin_summary():
        terminalreporter.write_line(line)
