"""Edge cases, closed forms and structural invariants of the CUDA path (GPU)."""
import math

import numpy as np
import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs

from kda_testutil import assert_close, check_full, oracle_full, run_gpu

pytestmark = pytest.mark.gpu
bf16, f32 = torch.bfloat16, torch.float32


def W(name, seed, H, B=1, T=0, lens=None, init=bf16, final=bf16, lb=-5.0, zero=False):
    if lens is not None:
        return Workload(name, seed, H=H, B=1, T=int(sum(lens)), seq_lens=list(lens), init_dtype=init,
                        final_dtype=final, lower_bound=lb, init_zero=zero)
    return Workload(name, seed, H=H, B=B, T=T, init_dtype=init, final_dtype=final, lower_bound=lb, init_zero=zero)


EDGE = [
    W("t1", 11, H=2, B=3, T=1),
    W("t31", 12, H=1, B=2, T=31, init=f32, final=bf16),
    W("t33", 13, H=1, B=1, T=33, init=bf16, final=f32),
    W("t64_noinit", 14, H=2, B=1, T=64, init=None, final=f32),
    W("empties", 15, H=2, lens=[0, 5, 0, 40, 0], init=f32, final=f32),
    W("one_seq_packed", 16, H=1, lens=[97], init=None, final=bf16),
    W("lb0", 17, H=2, B=1, T=96, lb=0.0),
    W("lb_limit", 18, H=2, B=1, T=130, lb=-5.45, init=f32, final=f32),
    W("h1_long_tail", 19, H=1, B=1, T=257, init=bf16, final=bf16),
]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_cases_against_oracle(w):
    inp = make_inputs(w, "cpu")
    out, final, bits = run_gpu(inp)
    assert bits == 0
    ref_out, ref_final = oracle_full(inp)
    check_full(inp, out, final, ref_out, ref_final)


def test_no_final_state():
    inp = make_inputs(W("nofinal", 20, H=2, B=1, T=70), "cpu")
    out, _, bits = run_gpu(inp, final_dtype=None)
    ref_out, _ = oracle_full(inp)
    check_full(inp, out, None, ref_out, None)


@pytest.mark.parametrize("dt", [f32, bf16])
def test_beta0_nodecay_keeps_state_bit_exact(dt):
    inp = make_inputs(W("closed1", 21, H=2, B=2, T=77, init=dt, final=dt, lb=0.0), "cpu")
    inp.beta.zero_()
    out, final, bits = run_gpu(inp)
    assert bits == 0
    assert torch.equal(final.cpu(), inp.initial_state), "state must be kept exactly"
    ref_out, _ = oracle_full(inp)
    check_full(inp, out, final, ref_out, inp.initial_state.double().numpy())


def test_beta1_nodecay_retrieves_v():
    H, T = 2, 64
    w = W("closed2", 22, H=H, B=1, T=T, init=f32, final=f32, lb=0.0)
    inp = make_inputs(w, "cpu")
    Hd = torch.tensor([[1.0]])
    while Hd.shape[0] < 128:
        Hd = torch.cat([torch.cat([Hd, Hd], 1), torch.cat([Hd, -Hd], 1)], 0)
    gen = torch.Generator().manual_seed(5)
    for h in range(H):
        rows = Hd[torch.randperm(128, generator=gen)[:T]]
        inp.k[0, :, h] = rows.to(bf16)
        inp.q[0, :, h] = rows.to(bf16)
    inp.beta.fill_(1.0)
    out, final, bits = run_gpu(inp)
    assert bits == 0
    expect = inp.scale * inp.v.double()
    assert_close("out == scale v", out.cpu().double().numpy(), expect.numpy(), bf16)


def test_packed_equals_separate_runs_bitwise():
    lens = [45, 0, 130, 64, 7]
    inp = make_inputs(W("pk", 23, H=3, lens=lens, init=f32, final=f32), "cuda")
    out, final, _ = run_gpu(inp)
    cu = [0] + list(np.cumsum(lens))
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.equal(final[n], inp.initial_state[n])
            continue
        sl = slice(cu[n], cu[n + 1])
        o1 = torch.empty_like(inp.q[:, sl])
        f1 = torch.empty_like(final[n:n + 1])
        kb.kda_fwd(inp.q[:, sl].contiguous(), inp.k[:, sl].contiguous(), inp.v[:, sl].contiguous(),
                   inp.g[:, sl].contiguous(), inp.beta[:, sl].contiguous(), inp.scale, o1, inp.A_log,
                   inp.dt_bias, inp.lower_bound, initial_state=inp.initial_state[n:n + 1].contiguous(),
                   final_state=f1)
        torch.cuda.synchronize()
        assert torch.equal(o1, out[:, sl]), f"sequence {n}: out differs from the packed run"
        assert torch.equal(f1[0], final[n]), f"sequence {n}: final state differs from the packed run"


def test_continuation_bitwise():
    T1, T2 = 96, 77
    inp = make_inputs(W("cont", 24, H=2, B=1, T=T1 + T2, init=f32, final=f32), "cuda")
    out, final, _ = run_gpu(inp)
    a = lambda t, s: t[:, s].contiguous()
    s1, s2 = slice(0, T1), slice(T1, T1 + T2)
    o1, o2 = torch.empty_like(a(inp.q, s1)), torch.empty_like(a(inp.q, s2))
    f1, f2 = torch.empty_like(final), torch.empty_like(final)
    kb.kda_fwd(a(inp.q, s1), a(inp.k, s1), a(inp.v, s1), a(inp.g, s1), a(inp.beta, s1), inp.scale, o1,
               inp.A_log, inp.dt_bias, inp.lower_bound, initial_state=inp.initial_state, final_state=f1)
    kb.kda_fwd(a(inp.q, s2), a(inp.k, s2), a(inp.v, s2), a(inp.g, s2), a(inp.beta, s2), inp.scale, o2,
               inp.A_log, inp.dt_bias, inp.lower_bound, initial_state=f1, final_state=f2)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([o1, o2], 1), out)
    assert torch.equal(f2, final)


@pytest.mark.parametrize("dt", [f32, bf16])
def test_inplace_alias_equals_separate_buffers(dt):
    inp = make_inputs(W("alias", 25, H=4, lens=[100, 33, 64], init=dt, final=dt), "cuda")
    out, final, _ = run_gpu(inp)
    state = inp.initial_state.clone()
    out2 = torch.full_like(out, float("nan"))
    _, _, bits = run_gpu(inp, out=out2, final=state, initial_state=state)
    assert bits == 0
    assert torch.equal(state, final)
    assert torch.equal(out2, out)


def test_repeat_runs_bitwise():
    inp = make_inputs(W("rep", 26, H=8, lens=[300, 17, 1000, 64], init=f32, final=f32), "cuda")
    o1, f1, _ = run_gpu(inp)
    o2, f2, _ = run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


@pytest.mark.parametrize("cu", [[1, 10, 20], [0, 15, 10], [0, 10, 21]])
def test_bad_cu_seqlens_sets_status_and_writes_nothing(cu):
    inp = make_inputs(W("badcu", 27, H=2, lens=[10, 10], init=f32, final=f32), "cuda")
    inp.cu_seqlens = torch.tensor(cu, dtype=torch.int64, device="cuda")
    out, final, bits = run_gpu(inp)
    assert bits & kb.KDA_DEVERR_CU_SEQLENS
    assert torch.isnan(out.float()).all()
    assert torch.isnan(final).all()


def test_partial_alias_rejected():
    inp = make_inputs(W("palias", 28, H=2, lens=[10, 10], init=f32, final=f32), "cuda")
    buf = torch.zeros(3 * 2 * 128 * 128, dtype=f32, device="cuda")
    init = buf[: 2 * 2 * 128 * 128].view(2, 2, 128, 128)
    fin = buf[2 * 128 * 128:].view(2, 2, 128, 128)
    with pytest.raises(kb.KDAError) as ei:
        run_gpu(inp, final=fin, initial_state=init)
    assert ei.value.status == kb.KDA_ERR_ALIAS


def test_lower_bound_outside_contract_rejected():
    inp = make_inputs(W("lbbad", 29, H=1, B=1, T=8, lb=-6.0), "cuda")
    with pytest.raises(kb.KDAError) as ei:
        run_gpu(inp)
    assert ei.value.status == kb.KDA_ERR_UNSUPPORTED


def test_canaries_after_buffers_untouched():
    w = W("canary", 30, H=2, lens=[50, 31], init=bf16, final=bf16)
    inp = make_inputs(w, "cuda")
    n_out = inp.q.numel()
    big = torch.full((n_out + 4096,), 3.0, dtype=bf16, device="cuda")
    out = big[:n_out].view_as(inp.q)
    n_st = 2 * 2 * 128 * 128
    bigs = torch.full((n_st + 4096,), 5.0, dtype=bf16, device="cuda")
    fin = bigs[:n_st].view(2, 2, 128, 128)
    _, _, bits = run_gpu(inp, out=out, final=fin)
    assert bits == 0
    assert (big[n_out:] == 3.0).all() and (bigs[n_st:] == 5.0).all()


def test_zero_length_batch():
    inp = make_inputs(W("t0", 31, H=2, B=2, T=0, init=f32, final=f32), "cuda")
    out, final, bits = run_gpu(inp)
    assert bits == 0
    assert torch.equal(final, inp.initial_state)


def test_forward_replays_from_a_cuda_graph():
    """kda_fwd is stream-ordered, allocates nothing and never synchronises, so a capture
    of one call replays it: new inputs copied into the captured buffers give the same
    results as an eager call on those inputs."""
    w = W("graph", 23, H=3, lens=[40, 0, 77, 33], init=f32, final=f32)
    a, b = make_inputs(w, "cpu"), make_inputs(W("graph", 24, H=3, lens=[40, 0, 77, 33], init=f32, final=f32), "cpu")
    dev = torch.device("cuda", 0)
    d = a.to(dev)
    out = torch.empty_like(d.q)
    final = torch.empty_like(d.initial_state)
    ws = torch.zeros(kb.kda_workspace_size(w.total_tokens, w.H, w.num_seqs), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def call():
        kb.kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, out, d.A_log, d.dt_bias, d.lower_bound,
                   initial_state=d.initial_state, final_state=final, cu_seqlens=d.cu_seqlens, workspace=ws,
                   stream=stream)

    with torch.cuda.stream(stream):
        call()                                    # warm-up outside the capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for src in (b, a):                            # replay on the other inputs, then on the first again
        for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
            getattr(d, name).copy_(getattr(src, name).to(dev))
        graph.replay()
        torch.cuda.synchronize()
        assert kb.kda_read_device_status(ws) == 0
        ref_out, ref_final, bits = run_gpu(src)
        assert bits == 0
        for row0, row1 in zip(src.cu_seqlens[:-1].tolist(), src.cu_seqlens[1:].tolist()):
            assert torch.equal(out[:, row0:row1].cpu(), ref_out[:, row0:row1].cpu())
        assert torch.equal(final.cpu(), ref_final.cpu())


@pytest.mark.parametrize("T", [1024, 4096])
def test_long_memory_keeps_state_precision(T):
    """Without decay (lower_bound = 0) the state remembers every token.  The fp32 state
    held in TMEM must stay within the fp32 tolerance over thousands of tokens; a state
    rounded to bf16 at every chunk boundary (KDA_KERNEL_BF16_STATE) drifts past it
    (tests/test_gpu_ablations.py)."""
    w = Workload(f"mem{T}", 31, H=4, B=1, T=T, init_dtype=f32, final_dtype=f32, lower_bound=0.0)
    inp = make_inputs(w, "cpu")
    inp.beta.mul_(0.2)   # moderate writes: the memory stays long
    out, final, bits = run_gpu(inp)
    assert bits == 0
    ref_out, ref_final = oracle_full(inp)
    check_full(inp, out, final, ref_out, ref_final)
