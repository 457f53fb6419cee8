"""Run only by the child process of tests/test_gpu_wait_timeout.py, against the test-only
build libkda_waittest.so (the file name keeps it out of the normal collection).

That build gives up a bounded wait after about 2 ms and, when KDA_TEST_SKIP_FULLD names a
chunk, has the inverse warp skip its FULLD arrival for that chunk: the chain's wait for it
runs out.  The call must come back with KDA_DEVERR_TIMEOUT set and the context must stay
usable: the next call, without the skip, matches the oracle.  The two ring schedules (two
CTAs per SM, one CTA per SM) are the ones exercised.
"""
import os

import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs

from kda_testutil import check_full, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


def _case(n_seqs, seed):
    lens = [70 + 13 * (i % 5) for i in range(n_seqs)]   # 3 chunks each, ragged tails
    return Workload(f"timeout{n_seqs}", seed, H=8, B=1, T=int(sum(lens)), seq_lens=lens,
                    init_dtype=torch.float32, final_dtype=torch.float32)


@pytest.mark.parametrize("n_seqs,schedule", [(20, kb.KDA_SCHEDULE_TWO_PER_SM), (9, kb.KDA_SCHEDULE_ONE_PER_SM)],
                         ids=["two_per_sm", "one_per_sm"])
def test_expired_wait_sets_the_timeout_bit_and_returns(n_seqs, schedule):
    assert os.path.basename(kb.library_path()) == "libkda_waittest.so"
    w = _case(n_seqs, 300 + n_seqs)
    if kb.kda_fwd_schedule(w.units) != schedule:
        pytest.skip("this GPU's SM count puts the case in another schedule")
    inp = make_inputs(w, "cpu")            # run_gpu copies these exact tensors to the device
    os.environ["KDA_TEST_SKIP_FULLD"] = "1"
    try:
        _, _, bits = run_gpu(inp)          # returns once every warp has wound down
    finally:
        del os.environ["KDA_TEST_SKIP_FULLD"]
    assert bits & kb.KDA_DEVERR_TIMEOUT
    out, final, bits = run_gpu(inp)        # the same context, no skip: a correct result
    assert bits == 0
    ref_out, ref_final = oracle_full(inp)
    check_full(inp, out, final, ref_out, ref_final)
