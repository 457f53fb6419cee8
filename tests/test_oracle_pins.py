"""Pins of the fp64 oracle against things other than itself (no GPU needed).

Each check is chosen so that a plausible mistake in the oracle (a dropped term, a
wrong sign or index, decay applied after the write, read-out before the write,
beta on the wrong side, a transposed state) fails at least one of them:

* an independent chunk-form evaluation (FlashInfer PR #4262 notes, sections 2-3:
  centered operands, L, Mqk, INV, Q_d, K_d, K_r, a, S_d, O_0, P, R, U, update),
  with chunk 16 and 32, centered and uncentered;
* brute force: the whole sequence as one materialised causal attention matrix
  with pairwise decays 2^(G_i - G_j) and one triangular solve;
* the transition-product form S_t = S_{t-1} diag(e^lambda_t)(I - beta k k^T) + beta v k^T;
* closed forms: beta = 0 with no decay keeps the state and reads a fixed memory;
  beta = 1 with no decay retrieves v exactly; beta = 0 with decay scales the state
  by exp(sum lambda) per key channel; two single-token steps worked by hand;
* structure: packed == independent runs, continuation == one run, V-channel
  permutation equivariance, empty sequences, untouched rows past cu_seqlens[N];
* the gate's range [lower_bound, 0] (its exact form is PARITY UNPINNED);
* the centering constants b and C printed for lower_bound = -5.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.linalg import solve_triangular

from oracle import kda_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LOG2E = 1.0 / math.log(2.0)
EPS = 1e-6


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(np.asarray(b)), 1e-300))


def gate_np(g, A_log, dt_bias, lb):
    # The gate reading (also used by the oracle); the pins below are about the recurrence.
    return lb / (1.0 + np.exp(-np.exp(A_log) * (g + dt_bias)))


def l2n(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + EPS)


def rand_unit(rng, T, K, V, lb=-5.0):
    return dict(
        q=rng.standard_normal((T, K)), k=rng.standard_normal((T, K)), v=rng.standard_normal((T, V)),
        g=rng.standard_normal((T, K)), beta=rng.uniform(0, 1, T), A_log=float(rng.uniform(0, 1)),
        dt_bias=rng.uniform(0, 1, K), lb=lb, S0=0.1 * rng.standard_normal((V, K)),
        scale=1.0 / math.sqrt(K))


def oracle_unit(u):
    """Run the oracle on one unit (B = 1, H = 1)."""
    T, K = u["q"].shape
    V = u["v"].shape[1]
    out, fin = O.kda_oracle_fwd(u["q"][None, :, None], u["k"][None, :, None], u["v"][None, :, None],
                                u["g"][None, :, None], u["beta"][None, :, None], u["scale"],
                                np.array([u["A_log"]]), u["dt_bias"][None], u["lb"],
                                initial_state=None if u["S0"] is None else u["S0"][None, None])
    return out[0, :, 0], fin[0, 0]


# ----------------------------------------------------------------------------
# Independent evaluations
# ----------------------------------------------------------------------------

def chunk_form(u, C=32, anchor="mid"):
    """Chunk form of the FlashInfer PR #4262 notes, sections 2 and 3, in fp64."""
    q, k, v, g, beta = u["q"], u["k"], u["v"], u["g"], u["beta"]
    T, K = q.shape
    V = v.shape[1]
    lam2 = gate_np(g, u["A_log"], u["dt_bias"], u["lb"]) * LOG2E       # base-2 log decay
    qh, kh = l2n(q), l2n(k)
    b = u["lb"] * LOG2E
    Cst = (C / 2) * b if anchor == "mid" else 0.0                      # fixed anchor (section 2)
    S = np.zeros((V, K)) if u["S0"] is None else u["S0"].copy()
    out = np.zeros((T, V))
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        sl = slice(c0, c0 + n)
        G = np.cumsum(lam2[sl], axis=0)                                # inclusive prefix
        GT = G[-1]
        Qc = u["scale"] * qh[sl] * np.exp2(G - Cst)
        Kc = kh[sl] * np.exp2(G - Cst)
        Ki = kh[sl] * np.exp2(Cst - G)
        L = np.tril(beta[sl, None] * (Kc @ Ki.T), -1)
        Mqk = np.tril(Qc @ Ki.T)
        INV = np.linalg.inv(np.eye(n) + L)
        Qd = u["scale"] * qh[sl] * np.exp2(G)
        Kd = kh[sl] * np.exp2(G)
        Kr = kh[sl] * np.exp2(GT - G)
        a = np.exp2(GT)
        Sd = S * a[None, :]
        O0 = S @ Qd.T
        P = S @ Kd.T
        R = (v[sl].T - P) * beta[sl][None, :]
        U = R @ INV.T
        S = Sd + U @ Kr
        out[sl] = (O0 + U @ Mqk.T).T
    return out, S


def materialised(u):
    """Whole sequence as one causal attention matrix with pairwise decays, one solve."""
    q, k, v, g, beta = u["q"], u["k"], u["v"], u["g"], u["beta"]
    T, K = q.shape
    V = v.shape[1]
    lam = gate_np(g, u["A_log"], u["dt_bias"], u["lb"])                 # natural log
    Gn = np.cumsum(lam, axis=0)
    qh, kh = l2n(q), l2n(k)
    S0 = np.zeros((V, K)) if u["S0"] is None else u["S0"]
    D = np.exp(Gn[:, None, :] - Gn[None, :, :])                         # [i, j, d] = e^(G_i - G_j)
    causal = np.tril(np.ones((T, T)), 0)
    strict = np.tril(np.ones((T, T)), -1)
    Wkk = np.einsum("id,jd,ijd->ij", kh, kh, np.where(causal[..., None] > 0, D, 0.0)) * strict
    Aqk = u["scale"] * np.einsum("id,jd,ijd->ij", qh, kh, np.where(causal[..., None] > 0, D, 0.0)) * causal
    Kd = kh * np.exp(Gn)
    rhs = beta[:, None] * (v - Kd @ S0.T)                               # [T, V]
    Ut = solve_triangular(np.eye(T) + beta[:, None] * Wkk, rhs, lower=True, unit_diagonal=True)
    out = u["scale"] * (qh * np.exp(Gn)) @ S0.T + Aqk @ Ut
    ST = S0 * np.exp(Gn[-1])[None, :] + Ut.T @ (kh * np.exp(Gn[-1][None, :] - Gn))
    return out, ST


def transition_product(u):
    """S_t = S_{t-1} diag(e^lambda_t) (I - beta_t kh kh^T) + beta_t v_t kh_t^T as explicit matrices."""
    q, k, v, g, beta = u["q"], u["k"], u["v"], u["g"], u["beta"]
    T, K = q.shape
    V = v.shape[1]
    lam = gate_np(g, u["A_log"], u["dt_bias"], u["lb"])
    qh, kh = l2n(q), l2n(k)
    S = np.zeros((V, K)) if u["S0"] is None else u["S0"].copy()
    out = np.zeros((T, V))
    for t in range(T):
        M = np.diag(np.exp(lam[t])) @ (np.eye(K) - beta[t] * np.outer(kh[t], kh[t]))
        S = S @ M + beta[t] * np.outer(v[t], kh[t])
        out[t] = u["scale"] * S @ qh[t]
    return out, S


# ----------------------------------------------------------------------------
# Agreement with the independent forms
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("T,K,V,C,anchor", [
    (70, 16, 8, 32, "mid"), (70, 16, 8, 32, "none"), (45, 16, 8, 16, "none"),
    (45, 16, 8, 16, "mid"), (33, 128, 128, 32, "mid"), (64, 128, 32, 32, "mid")])
def test_chunk_form_matches(T, K, V, C, anchor):
    rng = np.random.default_rng(1000 + T + K + C)
    u = rand_unit(rng, T, K, V)
    out, fin = oracle_unit(u)
    o2, f2 = chunk_form(u, C=C, anchor=anchor)
    assert rel(out, o2) < 1e-10
    assert rel(fin, f2) < 1e-10


@pytest.mark.parametrize("T,K,V,lb", [(1, 4, 3, -5.0), (7, 8, 8, -5.0), (16, 8, 6, -1.0),
                                      (40, 32, 16, -0.5), (64, 16, 16, -5.0)])
def test_materialised_matches(T, K, V, lb):
    rng = np.random.default_rng(2000 + T)
    u = rand_unit(rng, T, K, V, lb=lb)
    out, fin = oracle_unit(u)
    o2, f2 = materialised(u)
    assert rel(out, o2) < 1e-10
    assert rel(fin, f2) < 1e-10


def test_transition_product_matches():
    rng = np.random.default_rng(3000)
    for T, K, V in [(12, 8, 5), (30, 16, 16)]:
        u = rand_unit(rng, T, K, V, lb=-2.0)
        out, fin = oracle_unit(u)
        o2, f2 = transition_product(u)
        assert rel(out, o2) < 1e-11
        assert rel(fin, f2) < 1e-11


def test_no_initial_state_is_zero_state():
    rng = np.random.default_rng(3100)
    u = rand_unit(rng, 20, 8, 8)
    u0 = dict(u, S0=np.zeros((8, 8)))
    un = dict(u, S0=None)
    a, fa = oracle_unit(u0)
    b, fb = oracle_unit(un)
    assert np.array_equal(a, b) and np.array_equal(fa, fb)


# ----------------------------------------------------------------------------
# Closed forms
# ----------------------------------------------------------------------------

def test_beta0_nodecay_keeps_state_and_reads_fixed_memory():
    rng = np.random.default_rng(4000)
    u = rand_unit(rng, 50, 16, 12, lb=0.0)
    u["beta"] = np.zeros(50)
    out, fin = oracle_unit(u)
    assert np.array_equal(fin, u["S0"])                                 # exact
    expect = u["scale"] * l2n(u["q"]) @ u["S0"].T
    assert rel(out, expect) < 1e-13


def test_beta1_nodecay_retrieves_v():
    """beta = 1, no decay, q = k: out_t = scale v_t for any S0; with orthonormal
    keys every earlier (k_j, v_j) pair is still retrieved from the final state."""
    K = V = 16
    T = 12
    Hd = np.array([[1.0]])
    while Hd.shape[0] < K:
        Hd = np.block([[Hd, Hd], [Hd, -Hd]])                            # Sylvester-Hadamard rows
    rng = np.random.default_rng(4100)
    # Large-norm keys make the L2-norm epsilon negligible (relative 1e-6 / |k|^2).
    keys = 1024.0 * Hd[rng.permutation(K)[:T]]
    u = dict(q=keys.copy(), k=keys.copy(), v=rng.standard_normal((T, V)), g=rng.standard_normal((T, K)),
             beta=np.ones(T), A_log=0.3, dt_bias=rng.uniform(0, 1, K), lb=0.0,
             S0=rng.standard_normal((V, K)), scale=0.25)
    out, fin = oracle_unit(u)
    assert np.max(np.abs(out - 0.25 * u["v"])) < 1e-12
    kh = l2n(keys)
    assert np.max(np.abs(fin @ kh.T - u["v"].T)) < 1e-12
    # Orthogonal complement of the keys keeps S0's action.
    Q, _ = np.linalg.qr(np.concatenate([kh.T, rng.standard_normal((K, K - T))], axis=1))
    comp = Q[:, T:]
    assert np.max(np.abs(fin @ comp - u["S0"] @ comp)) < 1e-11


def test_beta0_decay_scales_columns():
    rng = np.random.default_rng(4200)
    u = rand_unit(rng, 37, 16, 8, lb=-0.7)
    u["beta"] = np.zeros(37)
    out, fin = oracle_unit(u)
    lam = gate_np(u["g"], u["A_log"], u["dt_bias"], u["lb"])
    cum = np.cumsum(lam, axis=0)
    assert rel(fin, u["S0"] * np.exp(cum[-1])[None, :]) < 1e-13
    expect = np.stack([u["scale"] * (u["S0"] * np.exp(cum[t])[None, :]) @ l2n(u["q"])[t] for t in range(37)])
    assert rel(out, expect) < 1e-13


def test_handworked_single_token():
    with open(os.path.join(GOLDEN, "t1_handworked.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        u = dict(q=np.array([c["q"]]), k=np.array([c["k"]]), v=np.array([c["v"]]),
                 g=np.array([c["g"]]), beta=np.array([c["beta"]]), A_log=c.get("A_log", 0.0),
                 dt_bias=np.array(c["dt_bias"]), lb=c["lower_bound"], S0=np.eye(2), scale=1.0)
        out, fin = oracle_unit(u)
        # eps = 1e-6 in the L2 norm perturbs the exact values by ~1e-7 relative.
        assert np.max(np.abs(out[0] - np.array(c["out"]))) < 1e-6, c["name"]
        assert np.max(np.abs(fin - np.array(c["final_state"]))) < 1e-6, c["name"]


# ----------------------------------------------------------------------------
# Structure
# ----------------------------------------------------------------------------

def _multi(rng, lens, H, K, V, init=True):
    Tt = int(sum(lens))
    d = dict(q=rng.standard_normal((1, Tt, H, K)), k=rng.standard_normal((1, Tt, H, K)),
             v=rng.standard_normal((1, Tt, H, V)), g=rng.standard_normal((1, Tt, H, K)),
             beta=rng.uniform(0, 1, (1, Tt, H)), A_log=rng.uniform(0, 1, H),
             dt_bias=rng.uniform(0, 1, (H, K)))
    S0 = 0.1 * rng.standard_normal((len(lens), H, V, K)) if init else None
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return d, S0, cu


def test_packed_equals_independent_runs():
    rng = np.random.default_rng(5000)
    lens = [5, 0, 33, 17, 64]
    H, K, V = 3, 8, 8
    d, S0, cu = _multi(rng, lens, H, K, V)
    out, fin = O.kda_oracle_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.3, d["A_log"], d["dt_bias"],
                                -3.0, initial_state=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        o1, f1 = O.kda_oracle_fwd(d["q"][:, sl], d["k"][:, sl], d["v"][:, sl], d["g"][:, sl],
                                  d["beta"][:, sl], 0.3, d["A_log"], d["dt_bias"], -3.0,
                                  initial_state=S0[n:n + 1])
        assert np.array_equal(out[:, sl], o1)
        assert np.array_equal(fin[n], f1[0])
    assert np.array_equal(fin[1], S0[1])            # empty sequence: final == initial


def test_batched_equals_packed():
    rng = np.random.default_rng(5100)
    B, T, H, K, V = 3, 21, 2, 8, 4
    d, _, _ = _multi(rng, [B * T], H, K, V, init=False)
    S0 = 0.1 * rng.standard_normal((B, H, V, K))
    args = (d["g"], d["beta"], 0.5, d["A_log"], d["dt_bias"], -5.0)
    resh = lambda x: x.reshape((B, T) + x.shape[2:])
    ob, fb = O.kda_oracle_fwd(resh(d["q"]), resh(d["k"]), resh(d["v"]), resh(d["g"]), resh(d["beta"]),
                              0.5, d["A_log"], d["dt_bias"], -5.0, initial_state=S0)
    cu = np.arange(0, B * T + 1, T, dtype=np.int64)
    op, fp = O.kda_oracle_fwd(d["q"], d["k"], d["v"], *args, initial_state=S0, cu_seqlens=cu)
    assert np.array_equal(ob.reshape(op.shape), op)
    assert np.array_equal(fb, fp)


def test_tokens_past_last_sequence_untouched():
    rng = np.random.default_rng(5200)
    d, S0, _ = _multi(rng, [40], 2, 8, 8)
    cu = np.array([0, 10, 25], dtype=np.int64)
    out, _ = O.kda_oracle_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 0.3, d["A_log"], d["dt_bias"],
                              -5.0, initial_state=S0[:1].repeat(2, 0), cu_seqlens=cu, out_fill=7.5)
    assert np.all(out[:, 25:] == 7.5)
    assert np.all(np.isfinite(out[:, :25]))


def test_continuation_equals_single_run():
    rng = np.random.default_rng(5300)
    u = rand_unit(rng, 70, 16, 8)
    out, fin = oracle_unit(u)
    a = {k: (v[:29] if isinstance(v, np.ndarray) and v.shape[:1] == (70,) else v) for k, v in u.items()}
    o1, f1 = oracle_unit(a)
    b = {k: (v[29:] if isinstance(v, np.ndarray) and v.shape[:1] == (70,) else v) for k, v in u.items()}
    b["S0"] = f1
    o2, f2 = oracle_unit(b)
    assert np.array_equal(np.concatenate([o1, o2]), out)
    assert np.array_equal(f2, fin)


def test_value_channel_permutation():
    rng = np.random.default_rng(5400)
    u = rand_unit(rng, 40, 16, 12)
    out, fin = oracle_unit(u)
    p = rng.permutation(12)
    up = dict(u, v=u["v"][:, p], S0=u["S0"][p])
    op, fp = oracle_unit(up)
    assert np.array_equal(op, out[:, p])
    assert np.array_equal(fp, fin[p])


def test_rejects_bad_cu_seqlens():
    rng = np.random.default_rng(5500)
    d, _, _ = _multi(rng, [10], 1, 4, 4, init=False)
    for cu in ([1, 10], [0, 6, 4], [0, 11]):
        with pytest.raises(ValueError):
            O.kda_oracle_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], 1.0, d["A_log"], d["dt_bias"],
                             -1.0, cu_seqlens=np.array(cu, dtype=np.int64))


# ----------------------------------------------------------------------------
# Gate range and centering constants
# ----------------------------------------------------------------------------

def test_gate_range_and_special_cases():
    rng = np.random.default_rng(6000)
    for _ in range(2000):
        g, A, dt = rng.standard_normal() * 6, rng.uniform(-2, 2), rng.uniform(-2, 2)
        lb = -rng.uniform(0, 8)
        lam = O.gate(g, A, dt, lb)
        assert lb <= lam <= 0.0
        assert O.gate(g, A, dt, 0.0) == 0.0
    # more gate input gives more decay (the reading is monotone in g)
    xs = np.linspace(-6, 6, 101)
    vals = [O.gate(x, 0.2, 0.1, -5.0) for x in xs]
    assert all(b <= a for a, b in zip(vals, vals[1:]))


def test_centering_constants():
    with open(os.path.join(GOLDEN, "centering_constants.json")) as f:
        c = json.load(f)
    b = c["lower_bound"] * LOG2E
    C = 16 * b
    assert round(b, c["b_printed_digits"]) == c["b"]
    assert round(C, c["C_printed_digits"]) == c["C"]
    # Centered exponents of a 32-token chunk stay within +-16|b|, the uncentered
    # radius of a 16-token chunk, for every prefix G in [32b, 0].
    for G in np.linspace(32 * b, 0, 257):
        assert abs(G - C) <= 16 * abs(b) + 1e-9
    # bf16 normal range (2^-126 .. 2^127) holds the centered factors iff 16|b| <= 126.
    lb_limit = -126.0 / (16 * LOG2E)
    assert abs(lb_limit - (-5.4585)) < 1e-4


# ----------------------------------------------------------------------------
# Interface variants (oracle flags): beta as a logit, the softplus gate
# ----------------------------------------------------------------------------

def _oracle_flags(u, flags):
    T, K = u["q"].shape
    V = u["v"].shape[1]
    out, fin = O.kda_oracle_fwd(u["q"][None, :, None], u["k"][None, :, None], u["v"][None, :, None],
                                u["g"][None, :, None], u["beta"][None, :, None], u["scale"],
                                np.array([u["A_log"]]), u["dt_bias"][None], u["lb"],
                                initial_state=None if u["S0"] is None else u["S0"][None, None], flags=flags)
    return out[0, :, 0], fin[0, 0]


def test_beta_logit_special_values():
    """sigmoid(0) = 1/2 exactly; sigmoid(40) = 1 to within 5e-18."""
    rng = np.random.default_rng(7000)
    u = rand_unit(rng, 23, 16, 8)
    for logit, value, tol in ((0.0, 0.5, 0.0), (40.0, 1.0, 1e-14)):
        ul = dict(u, beta=np.full(23, logit))
        uv = dict(u, beta=np.full(23, value))
        a, fa = _oracle_flags(ul, O.BETA_LOGIT)
        b, fb = _oracle_flags(uv, 0)
        assert rel(a, b) <= tol and rel(fa, fb) <= tol


def test_softplus_gate_special_values():
    """softplus(0) = ln 2, so g + dt_bias = 0 gives lambda = max(-exp(A_log) ln 2, lb);
    far below zero the gate vanishes, far above it sits on lower_bound; it is monotone."""
    assert O.gate_softplus(0.3, 0.0, -0.3, -5.0) == pytest.approx(-math.log(2.0), rel=1e-15)
    assert O.gate_softplus(-1.0, math.log(3.0), 1.0, -5.0) == pytest.approx(-3.0 * math.log(2.0), rel=1e-14)
    assert O.gate_softplus(0.0, math.log(3.0), 0.0, -1.5) == -1.5                # clamped
    assert -1e-20 < O.gate_softplus(-50.0, 0.0, 0.0, -5.0) < 0.0
    assert O.gate_softplus(50.0, 0.0, 0.0, -5.0) == -5.0
    rng = np.random.default_rng(7100)
    for _ in range(2000):
        g, A, dt = rng.standard_normal() * 6, rng.uniform(-2, 2), rng.uniform(-2, 2)
        lb = -rng.uniform(0, 8)
        assert lb <= O.gate_softplus(g, A, dt, lb) <= 0.0
    xs = np.linspace(-6, 6, 101)
    vals = [O.gate_softplus(x, 0.2, 0.1, -5.0) for x in xs]
    assert all(b <= a for a, b in zip(vals, vals[1:]))


def test_softplus_gate_decays_columns_by_ln2():
    """beta = 0 and g = -dt_bias everywhere: every channel decays by exp(-exp(A_log) ln 2)
    per token, so the final state is S0 (1/2)^(exp(A_log) T) column for column."""
    rng = np.random.default_rng(7200)
    T, K, V = 9, 16, 8
    u = rand_unit(rng, T, K, V, lb=-5.0)
    u["beta"] = np.zeros(T)
    u["g"] = -np.broadcast_to(u["dt_bias"], (T, K)).copy()
    _, fin = _oracle_flags(u, O.GATE_SOFTPLUS)
    assert rel(fin, u["S0"] * 0.5 ** (math.exp(u["A_log"]) * T)) < 1e-13
