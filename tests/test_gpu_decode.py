"""kda_decode: the single-token decode step, against the fp64 oracle.

One decode step is the recurrence of the oracle with one token per sequence (batched
mode, T = 1), so the oracle pins it directly.  Cases: fp32, bf16 and absent initial
states, the in-place update, a 64 x 64 batch, agreement with kda_fwd at T = 1, and 16
chained steps against the oracle run over the same 16 tokens.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs
from oracle.kda_oracle import kda_oracle_fwd

from kda_testutil import assert_close

pytestmark = pytest.mark.gpu


def _tok(t, i):
    """Token i of a batched [B, T, H, ...] tensor as [B, H, ...] (contiguous, on the GPU)."""
    return t[:, i].contiguous().cuda()


def _decode(inp, i, state, out_state=None):
    out = torch.full((inp.w.B, inp.w.H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kb.kda_decode(_tok(inp.q, i), _tok(inp.k, i), _tok(inp.v, i), _tok(inp.g, i), _tok(inp.beta, i), inp.scale, out,
                  inp.A_log.cuda(), inp.dt_bias.cuda(), inp.lower_bound, initial_state=state,
                  final_state=state if out_state is None else out_state)
    return out


def _oracle(inp, T):
    sl = lambda t: None if t is None else t[:, :T]
    return kda_oracle_fwd(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.g), sl(inp.beta), inp.scale, inp.A_log,
                          inp.dt_bias, inp.lower_bound, initial_state=inp.initial_state)


@pytest.mark.parametrize("sdtype", [torch.float32, torch.bfloat16, None], ids=["fp32", "bf16", "zero"])
def test_decode_step_matches_oracle(sdtype):
    w = Workload("dec_small", 61, H=3, B=5, T=1, init_dtype=sdtype, final_dtype=sdtype or torch.float32)
    inp = make_inputs(w, "cpu")
    ref_out, ref_final = _oracle(inp, 1)
    fdt = sdtype or torch.float32
    final = torch.full((w.B, w.H, 128, 128), float("nan"), dtype=fdt, device="cuda")
    init = inp.initial_state.cuda() if inp.initial_state is not None else None
    out = _decode(inp, 0, init, out_state=final)
    assert_close("decode out", out.double().cpu().numpy(), ref_out[:, 0], torch.bfloat16)
    assert_close("decode state", final.double().cpu().numpy(), ref_final, fdt)


def test_decode_in_place_batch_64x64():
    w = Workload("dec_64", 62, H=64, B=64, T=1, init_dtype=torch.float32, final_dtype=torch.float32)
    inp = make_inputs(w, "cpu")
    ref_out, ref_final = _oracle(inp, 1)
    state = inp.initial_state.cuda()
    out = _decode(inp, 0, state)
    assert_close("decode out", out.double().cpu().numpy(), ref_out[:, 0], torch.bfloat16)
    assert_close("decode state", state.double().cpu().numpy(), ref_final, torch.float32)


def test_decode_agrees_with_forward_at_one_token():
    w = Workload("dec_fwd", 63, H=4, B=6, T=1, init_dtype=torch.float32, final_dtype=torch.float32)
    inp = make_inputs(w, "cuda")
    out_f = torch.empty_like(inp.q)
    fin_f = torch.empty((w.B, w.H, 128, 128), dtype=torch.float32, device="cuda")
    kb.kda_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, out_f, inp.A_log, inp.dt_bias, inp.lower_bound,
               initial_state=inp.initial_state, final_state=fin_f)
    fin_d = torch.empty_like(fin_f)
    out_d = _decode(inp, 0, inp.initial_state, out_state=fin_d)
    assert_close("decode vs forward out", out_d.double().cpu().numpy(), out_f[:, 0].double().cpu().numpy(),
                 torch.bfloat16)
    assert_close("decode vs forward state", fin_d.double().cpu().numpy(), fin_f.double().cpu().numpy(),
                 torch.float32)


def test_sixteen_chained_steps_match_the_oracle():
    T = 16
    w = Workload("dec_chain", 64, H=4, B=3, T=T, init_dtype=torch.float32, final_dtype=torch.float32)
    inp = make_inputs(w, "cpu")
    ref_out, ref_final = _oracle(inp, T)
    state = inp.initial_state.cuda().clone()
    outs = [_decode(inp, i, state).double().cpu().numpy() for i in range(T)]
    assert_close("chained out", np.stack(outs, axis=1), ref_out, torch.bfloat16)
    assert_close("chained state", state.double().cpu().numpy(), ref_final, torch.float32)
