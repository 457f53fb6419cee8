"""The launch schedules of the prefill kernel, and that they do not change the numbers.

More (sequence, head) units than SMs run two CTAs to an SM; up to one unit per SM, one CTA
per SM; up to 7/25 as many units as SMs, a cluster of two CTAs per unit, and up to a quarter
as many a cluster of four (one CTA runs the recurrence over state resident in its Tensor
Memory, the others prepare chunks for it and push them into its shared memory).  A unit's
arithmetic is the same in each, so the same sequences must give bit-identical outputs and
final states whichever schedule their launch takes.  The cluster and one-CTA-per-SM launches
are also compared with the oracle over whole tensors, at and around the unit counts where the
schedule changes.
"""
import pytest
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Workload, make_inputs

from kda_testutil import check_full, oracle_full, run_gpu

pytestmark = pytest.mark.gpu
f32, bf16 = torch.float32, torch.bfloat16


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _cluster_max(kind=None, div=4):
    """The most units that still take a cluster schedule (every cluster resident at once)."""
    kind = kb.KDA_SCHEDULE_CLUSTER if kind is None else kind
    u = _sms() // div
    while u > 0 and kb.kda_fwd_schedule(u) != kind:
        u -= 1
    return u


def _cluster2_max():
    return _cluster_max(kb.KDA_SCHEDULE_CLUSTER2, 3)


def _prefix(inp, nseq):
    """The first `nseq` sequences of a packed input, as a packed input of their own."""
    w = inp.w
    lens = list(w.seq_lens[:nseq])
    T = int(sum(lens))
    sw = Workload(w.name + f"_first{nseq}", w.seed, H=w.H, B=1, T=T, seq_lens=lens, init_dtype=w.init_dtype,
                  final_dtype=w.final_dtype, lower_bound=w.lower_bound)
    sub = make_inputs(sw, "cpu")   # shapes and scalars; the tensors are replaced below
    for name in ("q", "k", "v", "g", "beta"):
        setattr(sub, name, getattr(inp, name)[:, :T].clone())
    sub.A_log, sub.dt_bias = inp.A_log.clone(), inp.dt_bias.clone()
    sub.scale, sub.lower_bound = inp.scale, inp.lower_bound
    sub.initial_state = None if inp.initial_state is None else inp.initial_state[:nseq].clone()
    sub.cu_seqlens = inp.cu_seqlens[: nseq + 1].clone()
    return sub


def _lens(n, seed):
    gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in torch.randint(1, 260, (n,), generator=gen)]
    lens[1] = 0            # an empty sequence
    lens[2] = 32           # exactly one chunk
    lens[3] = 65           # three chunks, the last of one token: every helper has work
    return lens


def test_schedule_thresholds():
    sms, cmax, cmax2 = _sms(), _cluster_max(), _cluster2_max()
    print(f"[schedule] SMs {sms}, clusters of four up to {cmax} units, of two up to {cmax2}")
    assert 1 <= cmax <= sms // 4 < cmax2 <= 7 * sms // 25
    want = lambda u: (kb.KDA_SCHEDULE_CLUSTER if u <= cmax else kb.KDA_SCHEDULE_CLUSTER2 if u <= cmax2 else
                      kb.KDA_SCHEDULE_ONE_PER_SM if u <= sms else kb.KDA_SCHEDULE_TWO_PER_SM)
    for u in sorted({1, 2, cmax, cmax + 1, sms // 4 + 1, cmax2, cmax2 + 1, sms // 2, sms // 2 + 1, sms - 1, sms,
                     sms + 1, 4 * sms}):
        assert kb.kda_fwd_schedule(u) == want(u), u
    assert kb.kda_fwd_schedule(0) == kb.KDA_SCHEDULE_TWO_PER_SM
    for flags in (kb.KDA_FLAG_BETA_LOGIT, kb.KDA_FLAG_GATE_SOFTPLUS):
        assert kb.kda_fwd_schedule(cmax, flags) == kb.KDA_SCHEDULE_CLUSTER
        assert kb.kda_fwd_schedule(cmax2, flags) == kb.KDA_SCHEDULE_CLUSTER2


def test_schedules_give_identical_numbers():
    """The first sequences of one packed input alone (the cluster of four), with more
    sequences (the cluster of two), more (one CTA per SM), and more again (two CTAs per SM)."""
    H, sms, cmax, cmax2 = 4, _sms(), _cluster_max(), _cluster2_max()
    n_cl = min(6, cmax // H)
    n_cl2 = cmax // H + 1                        # just past the clusters of four
    n_one = cmax2 // H + 1                       # just past the clusters of two
    n_two = sms // H + 1                         # past one unit per SM
    lens = _lens(n_two, 81)
    w = Workload("sched_same", 81, H=H, B=1, T=int(sum(lens)), seq_lens=lens, init_dtype=f32, final_dtype=f32)
    inp = make_inputs(w, "cpu")
    runs = {}
    for nseq in (n_cl, n_cl2, n_one, n_two):
        sub = _prefix(inp, nseq)
        runs[nseq] = (kb.kda_fwd_schedule(nseq * H),) + run_gpu(sub)
    assert [runs[n][0] for n in (n_cl, n_cl2, n_one, n_two)] == [
        kb.KDA_SCHEDULE_CLUSTER, kb.KDA_SCHEDULE_CLUSTER2, kb.KDA_SCHEDULE_ONE_PER_SM, kb.KDA_SCHEDULE_TWO_PER_SM]
    T_cl = int(sum(lens[:n_cl]))
    _, out_cl, fin_cl, bits_cl = runs[n_cl]
    assert bits_cl == 0
    for nseq in (n_cl2, n_one, n_two):
        _, out, fin, bits = runs[nseq]
        assert bits == 0
        torch.testing.assert_close(out[:, :T_cl].cpu(), out_cl.cpu(), rtol=0, atol=0, equal_nan=True)
        torch.testing.assert_close(fin[:n_cl].cpu(), fin_cl.cpu(), rtol=0, atol=0)


@pytest.mark.parametrize("units_kind", ["cluster_max", "cluster2_min", "cluster2_max", "one_per_sm_min", "one_per_sm"])
def test_schedule_against_oracle(units_kind):
    H, cmax, cmax2 = 1, _cluster_max(), _cluster2_max()
    nseq = {"cluster_max": cmax, "cluster2_min": cmax + 1, "cluster2_max": cmax2, "one_per_sm_min": cmax2 + 1,
            "one_per_sm": 100}[units_kind]
    lens = _lens(nseq, 82)
    w = Workload("sched_" + units_kind, 82, H=H, B=1, T=int(sum(lens)), seq_lens=lens, init_dtype=bf16,
                 final_dtype=f32)
    inp = make_inputs(w, "cpu")
    want = {"cluster_max": kb.KDA_SCHEDULE_CLUSTER, "cluster2_min": kb.KDA_SCHEDULE_CLUSTER2,
            "cluster2_max": kb.KDA_SCHEDULE_CLUSTER2}.get(units_kind, kb.KDA_SCHEDULE_ONE_PER_SM)
    assert kb.kda_fwd_schedule(w.units) == want
    out, final, bits = run_gpu(inp)
    assert bits == 0
    ref_out, ref_final = oracle_full(inp)
    check_full(inp, out, final, ref_out, ref_final)


@pytest.mark.parametrize("kind", ["four", "two"])
def test_cluster_schedule_long_sequences_and_variants(kind):
    """One long sequence per head (many rounds of the home's three slots and of the helpers'
    rings), every flag, in clusters of four and of two."""
    from oracle import kda_oracle as O
    from kda_testutil import assert_close
    H = 3 if kind == "four" else _cluster_max() + 2
    w = Workload("sched_long", 83, H=H, B=1, T=1000, seq_lens=[1000], init_dtype=f32, final_dtype=f32)
    inp = make_inputs(w, "cpu")
    assert kb.kda_fwd_schedule(w.units) == (kb.KDA_SCHEDULE_CLUSTER if kind == "four" else kb.KDA_SCHEDULE_CLUSTER2)
    for kflag, oflag in ((0, 0), (kb.KDA_FLAG_BETA_LOGIT | kb.KDA_FLAG_GATE_SOFTPLUS, O.BETA_LOGIT | O.GATE_SOFTPLUS)):
        ref_out, ref_final = O.kda_oracle_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.A_log,
                                              inp.dt_bias, inp.lower_bound, initial_state=inp.initial_state,
                                              cu_seqlens=inp.cu_seqlens, flags=oflag)
        d = inp.to(torch.device("cuda"))
        out = torch.zeros_like(d.q)
        final = torch.empty((1, w.H, 128, 128), dtype=f32, device="cuda")
        ws = kb.kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, out, d.A_log, d.dt_bias, d.lower_bound,
                        initial_state=d.initial_state, final_state=final, cu_seqlens=d.cu_seqlens, flags=kflag)
        assert kb.kda_read_device_status(ws) == 0
        assert_close("cluster out", out.double().cpu().numpy(), ref_out, bf16)
        assert_close("cluster state", final.double().cpu().numpy(), ref_final, f32)


def test_chain_trace_records_one_unit_without_changing_the_numbers():
    w = Workload("sched_trace", 84, H=2, B=1, T=500, seq_lens=[300, 200], init_dtype=f32, final_dtype=f32)
    assert kb.kda_fwd_schedule(w.units) == kb.KDA_SCHEDULE_CLUSTER
    inp = make_inputs(w, "cpu")
    out0, fin0, bits0 = run_gpu(inp)
    assert bits0 == 0
    n, h = 1, 1                                  # sequence 1 (200 tokens: 7 chunks), head 1
    nch = (200 + 31) // 32
    buf = torch.zeros((nch + 3, kb.KDA_TRACE_POINTS), dtype=torch.int64, device="cuda")
    kb.kda_fwd_set_trace(buf, unit=n * w.H + h)
    try:
        out1, fin1, bits1 = run_gpu(inp)
        # a launch on the two-CTA schedule leaves the buffer alone
        many = Workload("sched_trace_many", 85, H=64, B=4, T=40, init_dtype=None, final_dtype=f32)
        assert kb.kda_fwd_schedule(many.units) == kb.KDA_SCHEDULE_TWO_PER_SM
        snapshot = buf.clone()
        _, _, bits2 = run_gpu(make_inputs(many, "cpu"))
        assert bits2 == 0
        assert torch.equal(buf, snapshot)
    finally:
        kb.kda_fwd_set_trace(None)
    assert bits1 == 0
    torch.testing.assert_close(out1.cpu(), out0.cpu(), rtol=0, atol=0, equal_nan=True)
    torch.testing.assert_close(fin1.cpu(), fin0.cpu(), rtol=0, atol=0)
    t = buf.cpu()
    assert (t[:nch] > 0).all() and (t[nch:] == 0).all()
    for c in range(nch):
        r = t[c].tolist()
        assert r[0] <= r[4] <= r[5] <= r[6], r      # thread 0, in program order
        assert r[1] <= r[2] <= r[3] <= r[7], r      # the MMA warp, in program order
        # GEMM1 completes after its issue; GEMM2 issues after -R is in place.  (Point 6 is read
        # after thread 0's non-blocking arrival on the hand-off, so the MMA warp may pass the
        # barrier and stamp GEMM2's issue before thread 0 reads its clock: no order there.)
        assert r[3] < r[4] and r[5] <= r[7], r
    assert (t[1:nch, 0] > t[: nch - 1, 7]).all()    # chunks run in order
