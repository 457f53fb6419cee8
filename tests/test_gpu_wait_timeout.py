"""The timeout path of the bounded waits, on the GPU, in the form that faults nothing.

A test-only build (libkda_waittest.so: the sources compiled with -DKDA_WAIT_TEST) gives
up a wait after about 2 ms and can skip one producer arrival, chosen by the host.  In a
child process, a forward whose chain then waits in vain must return with
KDA_DEVERR_TIMEOUT set, every warp having wound down, and the next call on the same context
must be correct (tests/wait_timeout_cases.py).  The child has a hard time limit.
"""
import os
import subprocess
import sys

import pytest

from gated_delta_rule_36_gb300 import build as kbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_expired_wait_returns_the_timeout_status():
    lib = kbuild.build(variant="waittest")
    env = dict(os.environ, KDA_LIBRARY=lib)
    env.pop("KDA_TEST_SKIP_FULLD", None)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/wait_timeout_cases.py"], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
