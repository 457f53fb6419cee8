"""kda_fwd_host: the forward on host buffers, pipelined over groups of sequences.

The same kernels compute every (sequence, head) unit the same way whatever the group a
unit falls in, so the host entry point must reproduce kda_fwd on device copies of the
inputs bit for bit: outputs, final states, and the untouched rows of tokens outside
every sequence.  Cases: packed and batched requests, one to many groups (more groups
than sequences included), an in-place state, and a bf16 state.
"""
import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs

from kda_testutil import run_gpu

pytestmark = pytest.mark.gpu


def _pinned(t):
    return None if t is None else t.contiguous().pin_memory()


def _host_run(inp, groups, in_place=False):
    w = inp.w
    hq, hk, hv, hg, hb = (_pinned(t) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    ha, hd, hcu = _pinned(inp.A_log), _pinned(inp.dt_bias), _pinned(inp.cu_seqlens)
    hinit = _pinned(inp.initial_state.clone()) if inp.initial_state is not None else None
    hout = torch.full(hq.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    if in_place:
        hfinal = hinit
    else:
        hfinal = torch.full((w.num_seqs, w.H, w.V, w.K), float("nan"), dtype=w.final_dtype).pin_memory()
    nbytes = kb.kda_fwd_host_device_bytes(hq, cu_seqlens=hcu, initial_state=hinit, final_state=hfinal)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    kb.kda_fwd_host(hq, hk, hv, hg, hb, inp.scale, hout, ha, hd, inp.lower_bound, initial_state=hinit,
                    final_state=hfinal, cu_seqlens=hcu, device_buffer=buf, groups=groups, stream=stream)
    off = kb.kda_fwd_host_workspace_offset(hq, cu_seqlens=hcu, initial_state=hinit, final_state=hfinal)
    bits = kb.kda_read_device_status(buf.data_ptr() + off, stream)
    return hout, hfinal, bits


def _same(a, b):
    torch.testing.assert_close(a.cpu(), b.cpu(), rtol=0, atol=0, equal_nan=True)


CASES = [
    # packed, tokens past the last sequence (rows never written), an empty sequence
    (Workload("he_packed", 51, H=3, B=1, T=420, seq_lens=[200, 0, 64, 133, 7], init_dtype=torch.float32,
              final_dtype=torch.float32), (1, 2, 3, 16)),
    (Workload("he_batched", 52, H=2, B=3, T=75, init_dtype=torch.bfloat16, final_dtype=torch.bfloat16), (1, 2, 8)),
    (Workload("he_nostate", 53, H=4, B=1, T=300, seq_lens=[100, 150, 50], init_dtype=None,
              final_dtype=torch.float32), (3,)),
]


@pytest.mark.parametrize("w,groups", CASES, ids=["packed", "batched", "no_initial_state"])
def test_host_entry_matches_kda_fwd(w, groups):
    inp = make_inputs(w, "cpu")
    ref_out, ref_final, bits = run_gpu(inp)
    assert bits == 0
    for gcount in groups:
        out, final, hbits = _host_run(inp, gcount)
        assert hbits == 0
        _same(out, ref_out)
        _same(final, ref_final)


def test_host_entry_in_place_state():
    w = Workload("he_inplace", 54, H=2, B=1, T=260, seq_lens=[90, 170], init_dtype=torch.float32,
                 final_dtype=torch.float32)
    inp = make_inputs(w, "cpu")
    ref_out, ref_final, bits = run_gpu(inp)
    assert bits == 0
    out, final, hbits = _host_run(inp, 2, in_place=True)
    assert hbits == 0
    _same(out, ref_out)
    _same(final, ref_final)


def test_host_entry_from_another_thread():
    """The copy streams and events are kept per host thread: a call from a second thread
    uses its own and gives the same bits."""
    import threading
    w = CASES[0][0]
    inp = make_inputs(w, "cpu")
    ref_out, ref_final, bits = run_gpu(inp)
    assert bits == 0
    res = {}

    def work():
        try:
            res["r"] = _host_run(inp, 3)
        except Exception as exc:   # surfaced below
            res["e"] = exc

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert "e" not in res, res.get("e")
    out, final, hbits = res["r"]
    assert hbits == 0
    _same(out, ref_out)
    _same(final, ref_final)
