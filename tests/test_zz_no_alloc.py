"""kda_fwd_no_alloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin in a framework that owns the whole device pool and gives it
no allocator, a serving loop that must never allocate) cannot pass a workspace, so
this entry point uses an array built into the library instead.  The test calls it
through the C ABI twice in a row -- the second call runs on the array exactly as
the first call left it -- and checks that both results are bit-identical to kda_fwd
with a caller workspace: the same kernels run on the same inputs, only the workspace
differs.  It runs last so that a failure here cannot hide the others, and it passes
alone in a fresh process too.
"""
import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs

from kda_testutil import run_gpu

pytestmark = pytest.mark.gpu


def _no_alloc_run(inp):
    out = torch.full_like(inp.q, float("nan"))
    final = torch.full((inp.w.num_seqs, inp.w.H, 128, 128), float("nan"), dtype=inp.w.final_dtype,
                       device=inp.q.device)
    addr = kb.kda_fwd_no_alloc(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, out, inp.A_log, inp.dt_bias,
                               inp.lower_bound, initial_state=inp.initial_state, final_state=final,
                               cu_seqlens=inp.cu_seqlens)
    assert addr != 0
    assert kb.kda_read_device_status(addr) == 0
    return out, final


@pytest.mark.parametrize("w", [
    Workload("na_packed", 41, H=3, B=1, T=397, seq_lens=[200, 0, 64, 133], init_dtype=torch.float32,
             final_dtype=torch.float32),
    Workload("na_batched", 42, H=2, B=3, T=75, init_dtype=torch.bfloat16, final_dtype=torch.bfloat16),
], ids=["packed", "batched"])
def test_no_alloc_matches_kda_fwd_on_two_calls(w):
    inp = make_inputs(w, "cuda")
    ref_out, ref_final, bits = run_gpu(inp)
    assert bits == 0
    for _ in range(2):
        out, final = _no_alloc_run(inp)
        # rows outside every sequence keep the NaN fill on both sides: compare bit patterns
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), "out differs from kda_fwd"
        assert torch.equal(final, ref_final), "final_state differs from kda_fwd"


def test_no_alloc_rejects_too_many_sequences():
    n = 16384 + 1  # KDA_NO_ALLOC_MAX_SEQS + 1
    inp = make_inputs(Workload("na_many", 43, H=1, B=1, T=n, seq_lens=[1] * n, init_dtype=None,
                               final_dtype=torch.float32), "cuda")
    out = torch.empty_like(inp.q)
    with pytest.raises(kb.KDAError) as ei:
        kb.kda_fwd_no_alloc(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, out, inp.A_log, inp.dt_bias,
                            inp.lower_bound, cu_seqlens=inp.cu_seqlens)
    assert ei.value.status == kb.KDA_ERR_UNSUPPORTED
