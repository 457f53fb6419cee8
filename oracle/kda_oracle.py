"""ctypes front-end of the fp64 KDA oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this
module.  Inputs are widened exactly to float64 (bf16 and fp32 values are exactly
representable), the C code runs the token-by-token recurrence, and float64
results come back.

Which passages the recurrence follows, and the readings taken where the pages are
silent (gate form, L2-norm epsilon, packed-mode initial state), are listed in the
header of ``kda_oracle.c``.  The gate's exact form is PARITY UNPINNED.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (OpenMP over units)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            d = ctypes.c_double
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.kda_oracle_fwd.restype = ctypes.c_int
            lib.kda_oracle_fwd.argtypes = [i64, i64, i64, i64, i64, p, p, p, p, p, d, p, p, d,
                                           p, p, i64, p, p, ctypes.c_int]
            lib.kda_oracle_fwd_ex.restype = ctypes.c_int
            lib.kda_oracle_fwd_ex.argtypes = lib.kda_oracle_fwd.argtypes + [ctypes.c_uint]
            lib.kda_oracle_gate.restype = d
            lib.kda_oracle_gate.argtypes = [d, d, d, d]
            lib.kda_oracle_gate_softplus.restype = d
            lib.kda_oracle_gate_softplus.argtypes = [d, d, d, d]
            lib.kda_oracle_max_threads.restype = ctypes.c_int
            lib.kda_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach()
        if x.is_cuda:
            raise ValueError("the oracle takes host tensors only")
        x = x.to(dtype=__import__("torch").float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


BETA_LOGIT, GATE_SOFTPLUS = 0x1, 0x2   # kda_oracle_fwd_ex flags (interface variants)


def gate(g, A_log, dt_bias, lower_bound):
    """Scalar gate (natural log-decay), for tests of its range and special cases."""
    return _load().kda_oracle_gate(float(g), float(A_log), float(dt_bias), float(lower_bound))


def gate_softplus(g, A_log, dt_bias, lower_bound):
    """Scalar alternative gate max(-exp(A_log) softplus(g + dt_bias), lower_bound)."""
    return _load().kda_oracle_gate_softplus(float(g), float(A_log), float(dt_bias), float(lower_bound))


def max_threads() -> int:
    return int(_load().kda_oracle_max_threads())


def kda_oracle_fwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound,
                   initial_state=None, cu_seqlens=None, nthreads: int = 0,
                   out_fill: float = np.nan, flags: int = 0):
    """Run the oracle.  Shapes: q,k,g [B,T,H,K]; v [B,T,H,V]; beta [B,T,H];
    A_log [H]; dt_bias [H,K]; initial_state [Nseq,H,V,K] or None;
    cu_seqlens [N+1] (int64) or None.

    Returns (out [B,T,H,V] float64, final_state [Nseq,H,V,K] float64).  Rows of
    ``out`` outside every sequence keep ``out_fill``.
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    A_log, dt_bias = _f64(A_log), _f64(dt_bias)
    B, T, H, K = q.shape
    V = v.shape[3]
    assert k.shape == q.shape and g.shape == q.shape, "q, k, g must share a shape"
    assert v.shape[:3] == (B, T, H) and beta.shape == (B, T, H)
    assert A_log.shape == (H,) and dt_bias.shape == (H, K)
    cu = None
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        N = cu.shape[0] - 1
        nseq = N
    else:
        N = 0
        nseq = B
    S0 = _f64(initial_state)
    if S0 is not None:
        assert S0.shape == (nseq, H, V, K), f"initial_state shape {S0.shape}"
    out = np.full((B, T, H, V), out_fill, dtype=np.float64)
    final = np.empty((nseq, H, V, K), dtype=np.float64)
    rc = _load().kda_oracle_fwd_ex(B, T, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   float(scale), _ptr(A_log), _ptr(dt_bias), float(lower_bound),
                                   _ptr(S0), _ptr(cu), N, _ptr(out), _ptr(final), int(nthreads), int(flags))
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd rejected its arguments (code {rc})")
    return out, final
