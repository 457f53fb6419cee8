"""Interface variants (kda_fwd_ex / kda_decode_ex flags) against the fp64 oracle run with
the same flags: beta given as logits, the softplus gate, and both together.  The prefill
cases cover both kernel instantiations: few units (one CTA per SM) and 256 units (two CTAs
per SM); the decode cases use the batched one-token layout.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs
from oracle import kda_oracle as O

from kda_testutil import assert_close

pytestmark = pytest.mark.gpu

FLAGS = [(kb.KDA_FLAG_BETA_LOGIT, O.BETA_LOGIT), (kb.KDA_FLAG_GATE_SOFTPLUS, O.GATE_SOFTPLUS),
         (kb.KDA_FLAG_BETA_LOGIT | kb.KDA_FLAG_GATE_SOFTPLUS, O.BETA_LOGIT | O.GATE_SOFTPLUS)]
FLAG_IDS = ["beta_logit", "softplus_gate", "both"]


def _with_logit_beta(inp, seed):
    """beta ~ N(0, 1.5^2) logits (bf16), as a logit-beta caller would pass them."""
    gen = torch.Generator().manual_seed(seed)
    inp.beta = (1.5 * torch.randn(inp.beta.shape, generator=gen)).to(torch.bfloat16)
    return inp


WORKLOADS = [
    Workload("var_packed", 71, H=3, B=1, T=300, seq_lens=[100, 37, 0, 163], init_dtype=torch.float32,
             final_dtype=torch.float32),
    Workload("var_many_units", 72, H=64, B=1, T=4 * 70, seq_lens=[70, 70, 70, 70], init_dtype=torch.bfloat16,
             final_dtype=torch.bfloat16),
]


@pytest.mark.parametrize("w", WORKLOADS, ids=["few_units", "two_ctas_per_sm"])
@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_forward_variants_match_oracle(w, flags):
    kflag, oflag = flags
    inp = make_inputs(w, "cpu")
    if kflag & kb.KDA_FLAG_BETA_LOGIT:
        inp = _with_logit_beta(inp, w.seed)
    ref_out, ref_final = O.kda_oracle_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.A_log,
                                          inp.dt_bias, inp.lower_bound, initial_state=inp.initial_state,
                                          cu_seqlens=inp.cu_seqlens, flags=oflag)
    d = inp.to(torch.device("cuda"))
    out = torch.zeros_like(d.q)
    final = torch.empty((w.num_seqs, w.H, 128, 128), dtype=w.final_dtype, device="cuda")
    ws = kb.kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, out, d.A_log, d.dt_bias, d.lower_bound,
                    initial_state=d.initial_state, final_state=final, cu_seqlens=d.cu_seqlens, flags=kflag)
    assert kb.kda_read_device_status(ws) == 0
    covered = ~np.isnan(ref_out)
    assert_close("variant out", out.double().cpu().numpy()[covered], ref_out[covered], torch.bfloat16)
    assert_close("variant state", final.double().cpu().numpy(), ref_final, w.final_dtype)


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_decode_variants_match_oracle(flags):
    kflag, oflag = flags
    w = Workload("var_dec", 73, H=4, B=6, T=1, init_dtype=torch.float32, final_dtype=torch.float32)
    inp = make_inputs(w, "cpu")
    if kflag & kb.KDA_FLAG_BETA_LOGIT:
        inp = _with_logit_beta(inp, w.seed)
    ref_out, ref_final = O.kda_oracle_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.A_log,
                                          inp.dt_bias, inp.lower_bound, initial_state=inp.initial_state, flags=oflag)
    tok = lambda t: t[:, 0].contiguous().cuda()
    state = inp.initial_state.cuda().clone()
    out = torch.empty((w.B, w.H, 128), dtype=torch.bfloat16, device="cuda")
    kb.kda_decode(tok(inp.q), tok(inp.k), tok(inp.v), tok(inp.g), tok(inp.beta), inp.scale, out, inp.A_log.cuda(),
                  inp.dt_bias.cuda(), inp.lower_bound, initial_state=state, final_state=state, flags=kflag)
    assert_close("decode variant out", out.double().cpu().numpy(), ref_out[:, 0], torch.bfloat16)
    assert_close("decode variant state", state.double().cpu().numpy(), ref_final, torch.float32)


def test_unknown_flag_is_rejected():
    w = Workload("var_bad", 74, H=1, B=1, T=8, init_dtype=None, final_dtype=torch.float32)
    d = make_inputs(w, "cuda")
    out = torch.empty_like(d.q)
    with pytest.raises(kb.KDAError) as ei:
        kb.kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, out, d.A_log, d.dt_bias, d.lower_bound, flags=0x4)
    assert ei.value.status == kb.KDA_ERR_INVALID_ARG
