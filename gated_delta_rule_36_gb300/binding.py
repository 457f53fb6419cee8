"""Thin ctypes binding of the KDA C ABI (``include/kda.h``).

Argument marshalling only: every step of the forward runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
CPU fallback: if ``libkda.so`` is missing or the tensors are not on a CUDA device,
the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_ALIAS, KDA_ERR_WORKSPACE, KDA_ERR_CUDA = range(6)
KDA_BF16, KDA_F32, KDA_I64 = 0, 1, 2
KDA_DEVERR_CU_SEQLENS, KDA_DEVERR_TIMEOUT, KDA_DEVERR_INTERNAL = 0x1, 0x2, 0x4
HEAD_DIM = 128

# Every function include/kda.h declares.
EXPORTED = ("kda_workspace_size", "kda_fwd", "kda_status_string", "kda_last_error",
            "kda_read_device_status", "kda_fwd_no_alloc", "kda_fwd_host_device_bytes", "kda_fwd_host",
            "kda_fwd_host_workspace_offset", "kda_decode", "kda_fwd_ex", "kda_decode_ex", "kda_fwd_schedule",
            "kda_fwd_set_trace")
KDA_FLAG_BETA_LOGIT, KDA_FLAG_GATE_SOFTPLUS = 0x1, 0x2
KDA_FLAG_KERNEL_MASK = 0xF00
KDA_KERNEL_DEFAULT, KDA_KERNEL_CHUNK16, KDA_KERNEL_REGISTER_STATE, KDA_KERNEL_BF16_STATE = 0x000, 0x100, 0x200, 0x300
KDA_KERNEL_SMEM_STATE = 0x400
KDA_SCHEDULE_TWO_PER_SM, KDA_SCHEDULE_ONE_PER_SM, KDA_SCHEDULE_CLUSTER, KDA_SCHEDULE_CLUSTER2 = 0, 1, 2, 3
KDA_TRACE_POINTS = 8

_DTYPE = {torch.bfloat16: KDA_BF16, torch.float32: KDA_F32, torch.int64: KDA_I64}


class KdaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4)]


class KDAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return os.environ.get("KDA_LIBRARY") or _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load libkda.so (raises if it has not been built).  The environment variable
    KDA_LIBRARY names another build of the same ABI to load instead (the tests use it
    for the range-checked build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or os.environ.get("KDA_LIBRARY") or _build.LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"KDA CUDA library not found at {p}; build it with "
                              "gated_delta_rule_36_gb300.build.build()")
        lib = ctypes.CDLL(p)
        T = ctypes.POINTER(KdaTensor)
        lib.kda_workspace_size.restype = ctypes.c_size_t
        lib.kda_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.kda_fwd.restype = ctypes.c_int
        lib.kda_fwd.argtypes = [T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_float, T, T, T,
                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_fwd_set_trace.restype = ctypes.c_int
        lib.kda_fwd_set_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64]
        lib.kda_fwd_schedule.restype = ctypes.c_int
        lib.kda_fwd_schedule.argtypes = [ctypes.c_int64, ctypes.c_uint32, ctypes.POINTER(ctypes.c_int32)]
        lib.kda_read_device_status.restype = ctypes.c_int
        lib.kda_read_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.POINTER(ctypes.c_uint32)]
        lib.kda_fwd_no_alloc.restype = ctypes.c_int
        lib.kda_fwd_no_alloc.argtypes = [T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_float, T, T, T,
                                         ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
        lib.kda_fwd_ex.restype = ctypes.c_int
        lib.kda_fwd_ex.argtypes = [T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_float, T, T, T,
                                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_void_p]
        lib.kda_decode_ex.restype = ctypes.c_int
        lib.kda_decode_ex.argtypes = [T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_float, T, T,
                                      ctypes.c_uint32, ctypes.c_void_p]
        lib.kda_decode.restype = ctypes.c_int
        lib.kda_decode.argtypes = [T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_float, T, T, ctypes.c_void_p]
        lib.kda_fwd_host_device_bytes.restype = ctypes.c_size_t
        lib.kda_fwd_host_device_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                                  ctypes.c_int, ctypes.c_int]
        lib.kda_fwd_host_workspace_offset.restype = ctypes.c_size_t
        lib.kda_fwd_host_workspace_offset.argtypes = lib.kda_fwd_host_device_bytes.argtypes
        lib.kda_fwd_host.restype = ctypes.c_int
        lib.kda_fwd_host.argtypes = [T, T, T, T, T, ctypes.c_float, T, T, T, ctypes.c_float, T, T, T,
                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        if path is None:
            _lib = lib
        return lib


def _desc(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (the KDA path has no CPU fallback)")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.dim() > 4:
        raise ValueError(f"{name}: at most 4 dims")
    if t.dtype not in _DTYPE:
        raise ValueError(f"{name}: unsupported dtype {t.dtype}")
    d = KdaTensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or 16)
    d.dtype = _DTYPE[t.dtype]
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = int(s)
    return d


def _hdesc(t: Optional[torch.Tensor], name: str):
    """Descriptor of a host (CPU) tensor for kda_fwd_host."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name}: kda_fwd_host takes host tensors")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.dim() > 4 or t.dtype not in _DTYPE:
        raise ValueError(f"{name}: unsupported shape or dtype")
    d = KdaTensor()
    d.data = t.data_ptr() if t.numel() > 0 else (t.data_ptr() or 16)
    d.dtype = _DTYPE[t.dtype]
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = int(s)
    return d


def _state_code(t):
    return -1 if t is None else _DTYPE[t.dtype]


def kda_fwd_host_device_bytes(q, cu_seqlens=None, initial_state=None, final_state=None) -> int:
    """Device bytes kda_fwd_host needs for these (host) tensors."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    N = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else 0
    return int(load().kda_fwd_host_device_bytes(B, T, H, N, _state_code(initial_state), _state_code(final_state)))


def kda_fwd_host_workspace_offset(q, cu_seqlens=None, initial_state=None, final_state=None) -> int:
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    N = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else 0
    return int(load().kda_fwd_host_workspace_offset(B, T, H, N, _state_code(initial_state),
                                                    _state_code(final_state)))


def kda_fwd_host(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
                 final_state=None, cu_seqlens=None, device_buffer=None, groups=0, stream=None):
    """The forward on host tensors (pinned for asynchronous copies): copies in, computes
    and copies ``out`` / ``final_state`` back, pipelined over groups of sequences.
    ``device_buffer`` is a uint8 CUDA tensor of at least kda_fwd_host_device_bytes bytes.
    Returns once the work is enqueued on ``stream`` (torch's current stream by default)."""
    lib = load()
    descs = [_hdesc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (out, "out"),
                                       (A_log, "A_log"), (dt_bias, "dt_bias"), (initial_state, "initial_state"),
                                       (final_state, "final_state"), (cu_seqlens, "cu_seqlens"))]
    dq, dk, dv, dg, db, do, da, dd, di, df, dc = descs
    if device_buffer is None or not (isinstance(device_buffer, torch.Tensor) and device_buffer.is_cuda
                                     and device_buffer.dtype == torch.uint8):
        raise ValueError("device_buffer: must be a uint8 CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream(device_buffer.device)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = lib.kda_fwd_host(_ref(dq), _ref(dk), _ref(dv), _ref(dg), _ref(db), ctypes.c_float(float(scale)),
                          _ref(do), _ref(da), _ref(dd), ctypes.c_float(float(lower_bound)), _ref(di),
                          _ref(df), _ref(dc), ctypes.c_void_p(device_buffer.data_ptr()),
                          ctypes.c_size_t(device_buffer.numel()), ctypes.c_int(int(groups)), ctypes.c_void_p(sh))
    _check(lib, st)
    return device_buffer


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _check(lib, st: int):
    if st != KDA_OK:
        detail = lib.kda_last_error().decode()
        raise KDAError(st, f"{lib.kda_status_string(st).decode()}: {detail}")


def kda_workspace_size(T_total: int, H: int, N: int) -> int:
    return int(load().kda_workspace_size(int(T_total), int(H), int(N)))


def kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
            final_state=None, cu_seqlens=None, workspace=None, stream=None, flags=0):
    """Run the forward through the C ABI.  Tensors as in ``include/kda.h``.

    ``workspace`` (uint8 CUDA tensor) is allocated with torch when omitted;
    ``stream`` defaults to torch's current stream of q's device; ``flags`` (KDA_FLAG_*
    bits, plus one KDA_KERNEL_* value) selects the interface variants and the kernel
    through kda_fwd_ex.  Returns the workspace (its
    first word is the device status).
    """
    lib = load()
    descs = [_desc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (out, "out"),
                                      (A_log, "A_log"), (dt_bias, "dt_bias"), (initial_state, "initial_state"),
                                      (final_state, "final_state"), (cu_seqlens, "cu_seqlens"))]
    dq, dk, dv, dg, db, do, da, dd, di, df, dc = descs
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    nseq = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else B
    if workspace is None:
        workspace = torch.empty(kda_workspace_size(B * T, H, nseq), dtype=torch.uint8, device=q.device)
    if not (workspace.is_cuda and workspace.dtype == torch.uint8):
        raise ValueError("workspace: must be a uint8 CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    args = (_ref(dq), _ref(dk), _ref(dv), _ref(dg), _ref(db), ctypes.c_float(float(scale)),
            _ref(do), _ref(da), _ref(dd), ctypes.c_float(float(lower_bound)), _ref(di),
            _ref(df), _ref(dc), ctypes.c_void_p(workspace.data_ptr()), ctypes.c_size_t(workspace.numel()))
    if flags:
        st = lib.kda_fwd_ex(*args, ctypes.c_uint32(int(flags)), ctypes.c_void_p(sh))
    else:
        st = lib.kda_fwd(*args, ctypes.c_void_p(sh))
    _check(lib, st)
    return workspace


def kda_decode(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None, final_state=None,
               stream=None, flags=0):
    """One decode step (one token per sequence) through the C ABI: q, k, v, g, out
    [B, H, 128], beta [B, H], states [B, H, 128, 128]; final_state may be initial_state
    itself for the in-place update."""
    lib = load()
    descs = [_desc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (out, "out"),
                                      (A_log, "A_log"), (dt_bias, "dt_bias"), (initial_state, "initial_state"),
                                      (final_state, "final_state"))]
    dq, dk, dv, dg, db, do, da, dd, di, df = descs
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    args = (_ref(dq), _ref(dk), _ref(dv), _ref(dg), _ref(db), ctypes.c_float(float(scale)), _ref(do),
            _ref(da), _ref(dd), ctypes.c_float(float(lower_bound)), _ref(di), _ref(df))
    if flags:
        st = lib.kda_decode_ex(*args, ctypes.c_uint32(int(flags)), ctypes.c_void_p(sh))
    else:
        st = lib.kda_decode(*args, ctypes.c_void_p(sh))
    _check(lib, st)


def kda_fwd_set_trace(buffer=None, unit: int = 0) -> None:
    """Record the chain trace of (sequence, head) unit ``unit`` (sequence * H + head) into
    ``buffer`` (a CUDA int64 tensor of [chunks, KDA_TRACE_POINTS]) on later forward launches
    of this thread that take the cluster schedule; ``None`` turns it off."""
    lib = load()
    if buffer is None:
        _check(lib, lib.kda_fwd_set_trace(None, 0, 0))
        return
    if not (isinstance(buffer, torch.Tensor) and buffer.is_cuda and buffer.is_contiguous()):
        raise KDAError(KDA_ERR_INVALID_ARG, "trace buffer must be a contiguous CUDA tensor")
    _check(lib, lib.kda_fwd_set_trace(ctypes.c_void_p(buffer.data_ptr()), buffer.numel() * buffer.element_size(),
                                      int(unit)))


def kda_fwd_schedule(units: int, flags: int = 0) -> int:
    """KDA_SCHEDULE_* that kda_fwd takes on the current device for ``units`` (sequence, head)
    units: two CTAs per SM, one CTA per SM, or a cluster of four or of two CTAs per unit."""
    lib = load()
    sched = ctypes.c_int32(-1)
    _check(lib, lib.kda_fwd_schedule(int(units), int(flags), ctypes.byref(sched)))
    return int(sched.value)


def kda_read_device_status(workspace, stream=None) -> int:
    """Status bits of the last call that used ``workspace`` (a uint8 CUDA tensor, or
    the device address kda_fwd_no_alloc returns).  Synchronises the stream."""
    lib = load()
    if isinstance(workspace, torch.Tensor):
        addr, device = workspace.data_ptr(), workspace.device
    else:
        addr, device = int(workspace), torch.device("cuda", torch.cuda.current_device())
    if stream is None:
        stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    bits = ctypes.c_uint32(0)
    _check(lib, lib.kda_read_device_status(ctypes.c_void_p(addr), ctypes.c_void_p(sh), ctypes.byref(bits)))
    return int(bits.value)


def kda_fwd_no_alloc(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
                     final_state=None, cu_seqlens=None, stream=None) -> int:
    """kda_fwd for callers that cannot allocate device memory: the library uses its
    own fixed device array (KDA_NO_ALLOC_MAX_SEQS sequences at most) as the workspace
    and nothing is allocated.  Calls that overlap on the GPU share that array and
    race.  Returns the array's device address (for kda_read_device_status)."""
    lib = load()
    descs = [_desc(t, n) for t, n in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (out, "out"),
                                      (A_log, "A_log"), (dt_bias, "dt_bias"), (initial_state, "initial_state"),
                                      (final_state, "final_state"), (cu_seqlens, "cu_seqlens"))]
    dq, dk, dv, dg, db, do, da, dd, di, df, dc = descs
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    used = ctypes.c_void_p(0)
    st = lib.kda_fwd_no_alloc(_ref(dq), _ref(dk), _ref(dv), _ref(dg), _ref(db), ctypes.c_float(float(scale)),
                              _ref(do), _ref(da), _ref(dd), ctypes.c_float(float(lower_bound)), _ref(di),
                              _ref(df), _ref(dc), ctypes.c_void_p(sh), ctypes.byref(used))
    _check(lib, st)
    return int(used.value or 0)


def fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
        final_state=None, cu_seqlens=None):
    """FlashKDA-style convenience call: allocates the workspace, writes ``out`` and
    ``final_state`` in place and returns ``out``."""
    kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=initial_state,
            final_state=final_state, cu_seqlens=cu_seqlens)
    return out
