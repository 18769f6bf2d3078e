import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libraattn")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def pytest_terminal_summary(terminalreporter):
    """How many argmax rows the GPU tests compared, how many were near ties by the fp32
    score-error bound, and how many of those actually took the other key."""
    parity = sys.modules.get("parity")
    if parity is None or not parity.ARGMAX_LOG:
        return
    rows = sum(r for _, r, _, _ in parity.ARGMAX_LOG)
    near = sum(n for _, _, n, _ in parity.ARGMAX_LOG)
    diff = sum(d for _, _, _, d in parity.ARGMAX_LOG)
    terminalreporter.write_line(f"argmax: {rows} rows compared in {len(parity.ARGMAX_LOG)} checks; "
                                f"{near} near ties within the fp32 score-error bound; {diff} rows took the other key")
    for what, r, n, d in parity.ARGMAX_LOG:
        if d:
            terminalreporter.write_line(f"  {what}: {d} of {r} rows differ ({n} near ties)")
