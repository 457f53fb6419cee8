"""Shared helpers of the GPU tests: run the CUDA path through the C ABI, run the
oracle on the same seeded inputs, and compare within the stated tolerances.

Tolerances (whole compared tensor): bf16 out and bf16 state: max |diff| <= 2e-2
and relative Frobenius <= 1e-2; fp32 state: relative Frobenius <= 5e-3.
cu_seqlens indexing is checked bit-exactly: rows outside every sequence keep a
NaN sentinel.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300.inputs import Inputs
from oracle import kda_oracle as O

BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 1e-2
F32_REL_FRO = 5e-3

# (test, tensor, dtype, max |diff|, relative Frobenius, compared elements) of every
# whole-tensor comparison of a full-size workload; conftest prints it after the run
PARITY_LOG = []


def run_gpu(inp: Inputs, final_dtype=None, out=None, final=None, workspace=None, initial_state="same", flags=0):
    """Run the CUDA path (``flags``: KDA_FLAG_* / KDA_KERNEL_* of kda_fwd_ex).  Returns
    (out, final_state, device status bits) on the device."""
    w = inp.w
    dev = torch.device("cuda")
    d = inp if inp.q.is_cuda else inp.to(dev)
    if out is None:
        out = torch.full_like(d.q, float("nan"))
    fd = final_dtype or w.final_dtype
    if final is None and fd is not None:
        final = torch.full((w.num_seqs, w.H, w.V, w.K), float("nan"), dtype=fd, device=dev)
    init = d.initial_state if isinstance(initial_state, str) else initial_state
    ws = kb.kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.scale, out, d.A_log, d.dt_bias, d.lower_bound,
                    initial_state=init, final_state=final, cu_seqlens=d.cu_seqlens, workspace=workspace,
                    flags=flags)
    bits = kb.kda_read_device_status(ws)
    return out, final, bits


def seq_bounds(w):
    if w.packed:
        cu = np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int64)
        return [(int(cu[n]), int(cu[n + 1])) for n in range(len(w.seq_lens))]
    return [(b * w.T, (b + 1) * w.T) for b in range(w.B)]


def oracle_units(inp: Inputs, units, nthreads=0):
    """Oracle on selected (sequence, head) units.  Returns {(n, h): (out [len,V], final [V,K])}."""
    w = inp.w
    cpu = (lambda t: None if t is None else t.detach().cpu()) if inp.q.is_cuda else (lambda t: t)
    bounds = seq_bounds(w)
    heads = sorted({h for _, h in units})
    seqs = sorted({n for n, _ in units})
    res = {}
    flat = lambda t: t.reshape((w.B * w.T,) + tuple(t.shape[2:]))
    q, k, v, g, beta = (flat(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    A_log, dt_bias = cpu(inp.A_log), cpu(inp.dt_bias)
    for n in seqs:
        bos, eos = bounds[n]
        hs = [h for (m, h) in units if m == n]
        hi = torch.tensor(hs, device=q.device)
        sl = lambda t: cpu(t[bos:eos].index_select(1, hi)).unsqueeze(0)
        S0 = None
        if inp.initial_state is not None:
            S0 = cpu(inp.initial_state[n].index_select(0, hi.to(inp.initial_state.device))).unsqueeze(0)
        o, f = O.kda_oracle_fwd(sl(q), sl(k), sl(v), sl(g), sl(beta), inp.scale,
                                A_log[hs], dt_bias[hs], inp.lower_bound, initial_state=S0,
                                nthreads=nthreads)
        for j, h in enumerate(hs):
            res[(n, h)] = (o[0, :, j], f[0, j])
    return res


def oracle_full(inp: Inputs, nthreads=0):
    cpu = lambda t: None if t is None else t.detach().cpu()
    return O.kda_oracle_fwd(cpu(inp.q), cpu(inp.k), cpu(inp.v), cpu(inp.g), cpu(inp.beta), inp.scale,
                            cpu(inp.A_log), cpu(inp.dt_bias), inp.lower_bound,
                            initial_state=cpu(inp.initial_state), cu_seqlens=cpu(inp.cu_seqlens),
                            nthreads=nthreads)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)) if d.size else 0.0
    return max_abs, rel


def assert_close(name, got, ref, dtype):
    got = got.detach().float().cpu().numpy() if isinstance(got, torch.Tensor) else got
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    max_abs, rel = errors(got, ref)
    if os.environ.get("KDA_TEST_VERBOSE"):
        print(f"[err] {name}: max_abs={max_abs:.3e} rel_fro={rel:.3e} ({'fp32' if dtype == torch.float32 else 'bf16'})")
    if dtype == torch.float32:
        assert rel <= F32_REL_FRO, f"{name}: rel Frobenius {rel:.3e} > {F32_REL_FRO}"
    else:
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_FRO, \
            f"{name}: max abs {max_abs:.3e} (<= {BF16_MAX_ABS}), rel Frobenius {rel:.3e} (<= {BF16_REL_FRO})"
    return max_abs, rel


def check_full(inp: Inputs, out, final, ref_out, ref_final):
    """Whole-tensor comparison plus the bit-exact check of untouched rows."""
    w = inp.w
    o = out.detach().float().cpu().numpy()
    covered = np.zeros((w.B, w.T), dtype=bool)
    for (bos, eos) in seq_bounds(w):
        covered.reshape(-1)[bos:eos] = True
    assert np.all(np.isnan(o[~covered])), "rows outside every sequence were written"
    stats = {"out": assert_close("out", o[covered], ref_out[covered], torch.bfloat16)}
    if final is not None:
        stats["final"] = assert_close("final_state", final, ref_final, final.dtype)
    return stats


def check_units(inp: Inputs, out, final, ref_units):
    w = inp.w
    bounds = seq_bounds(w)
    of = out.reshape(w.B * w.T, w.H, w.V)
    stats = {}
    for (n, h), (ro, rf) in ref_units.items():
        bos, eos = bounds[n]
        stats[(n, h, "out")] = assert_close(f"out[seq {n}, head {h}]", of[bos:eos, h], ro, torch.bfloat16)
        if final is not None:
            stats[(n, h, "final")] = assert_close(f"final[seq {n}, head {h}]", final[n, h], rf, final.dtype)
    return stats


class _Acc:
    """Running max |diff|, sum diff^2 and sum ref^2 over the pieces of one tensor."""

    def __init__(self):
        self.max_abs, self.d2, self.r2, self.n = 0.0, 0.0, 0.0, 0

    def add(self, got, ref):
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        assert np.all(np.isfinite(got)), "non-finite values"
        d = got - ref
        if d.size:
            self.max_abs = max(self.max_abs, float(np.max(np.abs(d))))
        self.d2 += float(np.sum(d * d))
        self.r2 += float(np.sum(ref * ref))
        self.n += d.size

    def rel(self):
        return math.sqrt(self.d2) / max(math.sqrt(self.r2), 1e-30)


def _verdict(label, name, acc, dtype):
    rel = acc.rel()
    kind = "fp32" if dtype == torch.float32 else "bf16"
    PARITY_LOG.append((label, name, kind, acc.max_abs, rel, acc.n))
    if os.environ.get("KDA_TEST_VERBOSE"):
        print(f"[err] {label} {name}: max_abs={acc.max_abs:.3e} rel_fro={rel:.3e} ({kind}, {acc.n} elements)")
    if dtype == torch.float32:
        assert rel <= F32_REL_FRO, f"{label} {name}: rel Frobenius {rel:.3e} > {F32_REL_FRO}"
    else:
        assert acc.max_abs <= BF16_MAX_ABS and rel <= BF16_REL_FRO, \
            f"{label} {name}: max abs {acc.max_abs:.3e} (<= {BF16_MAX_ABS}), rel Frobenius {rel:.3e} (<= {BF16_REL_FRO})"


def check_whole_by_sequence(inp: Inputs, out, final, label, nthreads=0):
    """Whole-tensor comparison of a full-size run with the oracle, one sequence at a time.

    The oracle runs every head of one sequence per call (its OpenMP loop is over the
    heads), so host memory stays bounded by one sequence's fp64 copies however large the
    workload.  max |diff| and the relative Frobenius error are accumulated over the whole
    of ``out`` (every row that belongs to a sequence) and the whole of ``final``; rows
    outside every sequence must keep their NaN sentinel, bit for bit."""
    w = inp.w
    cpu = lambda t: None if t is None else t.detach().cpu()
    flat = lambda t: t.reshape((w.B * w.T,) + tuple(t.shape[2:]))
    q, k, v, g, beta = (flat(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    of = flat(out)
    A_log, dt_bias = cpu(inp.A_log), cpu(inp.dt_bias)
    acc_o, acc_f = _Acc(), _Acc()
    bounds = seq_bounds(w)
    for n, (bos, eos) in enumerate(bounds):
        sl = lambda t: cpu(t[bos:eos]).unsqueeze(0)
        S0 = None if inp.initial_state is None else cpu(inp.initial_state[n]).unsqueeze(0)
        ro, rf = O.kda_oracle_fwd(sl(q), sl(k), sl(v), sl(g), sl(beta), inp.scale, A_log, dt_bias,
                                  inp.lower_bound, initial_state=S0, nthreads=nthreads)
        acc_o.add(cpu(of[bos:eos]).double().numpy(), ro[0])
        if final is not None:
            acc_f.add(cpu(final[n]).double().numpy(), rf[0])
    covered = torch.zeros(w.B * w.T, dtype=torch.bool)
    for bos, eos in bounds:
        covered[bos:eos] = True
    outside = cpu(of)[~covered]
    assert torch.isnan(outside.float()).all(), "rows outside every sequence were written"
    _verdict(label, "out", acc_o, torch.bfloat16)
    if final is not None:
        _verdict(label, "final_state", acc_f, final.dtype)
    return acc_o, acc_f
