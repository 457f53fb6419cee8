"""The range-checked build (libkda_checked.so, the sources compiled with -DKDA_CHECKED).

It checks the indices that depend on the data or the thread (global state rows, beta and
output rows, token coordinates of the tensor copies, the tile index functions' arguments);
a bad one sets KDA_DEVERR_INTERNAL and is clamped into range instead of faulting.  The
small workloads and the edge cases run against it in a child process (the variable
KDA_LIBRARY makes the binding load it there): every result must match the oracle and no
status bit may be set.
"""
import os
import subprocess
import sys

import pytest

from gated_delta_rule_36_gb300 import build as kbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_passes_the_parity_cases():
    lib = kbuild.build(variant="checked")
    env = dict(os.environ, KDA_LIBRARY=lib)
    cases = ["tests/test_gpu_parity.py::test_small_workloads_whole_tensor",
             "tests/test_gpu_invariants.py::test_edge_cases_against_oracle",
             "tests/test_gpu_invariants.py::test_packed_equals_separate_runs_bitwise",
             "tests/test_gpu_schedules.py",
             "tests/checked_build_identity.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *cases],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
