import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU case")


def pytest_terminal_summary(terminalreporter):
    """After the run: the error figures of every whole-tensor comparison of a full-size
    workload (max |diff| and relative Frobenius error against the fp64 oracle)."""
    try:
        from kda_testutil import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle (whole tensors)")
    for label, name, kind, max_abs, rel, n in PARITY_LOG:
        tr.write_line(f"{label:>22s} {name:<12s} {kind}: max|d| {max_abs:.3e}  rel-Fro {rel:.3e}  ({n} elements)")
