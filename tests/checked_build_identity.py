"""Run only by the child process of tests/test_gpu_checked.py (the file name keeps it out of
the normal collection): the library the binding loaded there is the range-checked build."""
import os

import pytest

from gated_delta_rule_36_gb300 import binding as kb

pytestmark = pytest.mark.gpu


def test_loaded_library_is_the_checked_build():
    assert os.environ.get("KDA_LIBRARY"), "run through tests/test_gpu_checked.py"
    assert kb.load()._name == os.environ["KDA_LIBRARY"]
    assert os.path.basename(kb.library_path()) == "libkda_checked.so"
