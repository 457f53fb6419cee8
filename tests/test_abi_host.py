"""Host-only checks of the C ABI (no GPU, no compute calls).

The library must build for sm_103a, load, and export every function
``include/kda.h`` declares.  Invalid requests must be rejected with the right
status before anything is enqueued, so these calls use fake device addresses.
"""
import ctypes
import os
import re

import pytest

from gated_delta_rule_36_gb300 import binding as kb
from gated_delta_rule_36_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kb.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert set(declared_functions()) == set(kb.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_size(lib):
    assert kb.kda_workspace_size(0, 1, 0) >= 256 + 4
    assert kb.kda_workspace_size(2048, 96, 3) >= 256 + 3 * 4
    assert kb.kda_workspace_size(270000, 64, 64) % 256 == 0
    assert lib.kda_workspace_size(-1, 1, 1) == 0


def test_status_strings(lib):
    for s in range(6):
        assert lib.kda_status_string(s)


BASE = 0x7F0000000000  # fake, 256-byte aligned device addresses: never dereferenced


def T(dtype, shape, addr):
    d = kb.KdaTensor()
    d.data = addr
    d.dtype = dtype
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = s
    return d


def args(**over):
    B, Tn, H = over.pop("BTH", (1, 64, 2))
    a = dict(
        q=T(kb.KDA_BF16, (B, Tn, H, 128), BASE + 0x0000000),
        k=T(kb.KDA_BF16, (B, Tn, H, 128), BASE + 0x1000000),
        v=T(kb.KDA_BF16, (B, Tn, H, 128), BASE + 0x2000000),
        g=T(kb.KDA_BF16, (B, Tn, H, 128), BASE + 0x3000000),
        beta=T(kb.KDA_BF16, (B, Tn, H), BASE + 0x4000000),
        out=T(kb.KDA_BF16, (B, Tn, H, 128), BASE + 0x5000000),
        A_log=T(kb.KDA_F32, (H,), BASE + 0x6000000),
        dt_bias=T(kb.KDA_F32, (H, 128), BASE + 0x7000000),
        init=None, final=None, cu=None, scale=0.088, lb=-5.0,
        ws=BASE + 0x9000000, ws_bytes=1 << 20)
    a.update(over)
    return a


def call(lib, **over):
    a = args(**over)
    r = lambda d: None if d is None else ctypes.byref(d)
    return lib.kda_fwd(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]), ctypes.c_float(a["scale"]),
                       r(a["out"]), r(a["A_log"]), r(a["dt_bias"]), ctypes.c_float(a["lb"]), r(a["init"]),
                       r(a["final"]), r(a["cu"]), ctypes.c_void_p(a["ws"]), ctypes.c_size_t(a["ws_bytes"]),
                       ctypes.c_void_p(0))


def test_rejections(lib):
    st = lambda d, H=2: T(d, (1, H, 128, 128), BASE + 0x8000000)
    cases = [
        (dict(q=T(kb.KDA_F32, (1, 64, 2, 128), BASE)), kb.KDA_ERR_INVALID_ARG),
        (dict(q=T(kb.KDA_BF16, (1, 64, 2, 64), BASE)), kb.KDA_ERR_UNSUPPORTED),
        (dict(q=None), kb.KDA_ERR_INVALID_ARG),
        (dict(k=T(kb.KDA_BF16, (1, 63, 2, 128), BASE + 0x1000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(beta=T(kb.KDA_BF16, (1, 64, 3), BASE + 0x4000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(A_log=T(kb.KDA_BF16, (2,), BASE + 0x6000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(dt_bias=T(kb.KDA_F32, (2, 64), BASE + 0x7000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(lb=0.5), kb.KDA_ERR_INVALID_ARG),
        (dict(lb=float("nan")), kb.KDA_ERR_INVALID_ARG),
        (dict(lb=-6.0), kb.KDA_ERR_UNSUPPORTED),
        (dict(scale=float("inf")), kb.KDA_ERR_INVALID_ARG),
        (dict(q=T(kb.KDA_BF16, (1, 64, 2, 128), BASE + 8)), kb.KDA_ERR_INVALID_ARG),
        (dict(init=T(kb.KDA_F32, (1, 2, 128, 64), BASE + 0x8000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(final=T(kb.KDA_I64, (1, 2, 128, 128), BASE + 0x8000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(init=st(kb.KDA_F32), final=T(kb.KDA_F32, (1, 2, 128, 128), BASE + 0x8000000 + 4096)),
         kb.KDA_ERR_ALIAS),
        (dict(init=st(kb.KDA_F32), final=st(kb.KDA_BF16)), kb.KDA_ERR_ALIAS),
        (dict(BTH=(2, 32, 2), cu=T(kb.KDA_I64, (3,), BASE + 0xA000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(cu=T(kb.KDA_F32, (3,), BASE + 0xA000000)), kb.KDA_ERR_INVALID_ARG),
        (dict(cu=T(kb.KDA_I64, (3,), BASE + 0xA000000), init=st(kb.KDA_F32)), kb.KDA_ERR_INVALID_ARG),
        (dict(ws=BASE + 0x9000000 + 16), kb.KDA_ERR_WORKSPACE),
        (dict(ws=0), kb.KDA_ERR_WORKSPACE),
        (dict(ws_bytes=16), kb.KDA_ERR_WORKSPACE),
    ]
    for over, expect in cases:
        got = call(lib, **over)
        assert got == expect, (over, got, lib.kda_last_error())
        assert lib.kda_last_error(), over


def test_kernel_field_rejections(lib):
    """The kernel field of kda_fwd_ex's flags: one listed value at a time, and no interface
    flag beside a kernel other than the default; refused before anything is enqueued."""
    a = args()
    r = lambda t: None if t is None else ctypes.byref(t)

    def call_ex(flags):
        return lib.kda_fwd_ex(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]), ctypes.c_float(a["scale"]),
                              r(a["out"]), r(a["A_log"]), r(a["dt_bias"]), ctypes.c_float(a["lb"]), r(a["init"]),
                              r(a["final"]), r(a["cu"]), ctypes.c_void_p(a["ws"]), ctypes.c_size_t(16),
                              ctypes.c_uint32(flags), ctypes.c_void_p(0))

    assert call_ex(0xF00) == kb.KDA_ERR_INVALID_ARG
    assert call_ex(0x500) == kb.KDA_ERR_INVALID_ARG
    assert call_ex(0x4) == kb.KDA_ERR_INVALID_ARG
    assert call_ex(0x1000) == kb.KDA_ERR_INVALID_ARG
    for kern in (kb.KDA_KERNEL_CHUNK16, kb.KDA_KERNEL_REGISTER_STATE, kb.KDA_KERNEL_BF16_STATE,
                 kb.KDA_KERNEL_SMEM_STATE):
        assert call_ex(kern | kb.KDA_FLAG_BETA_LOGIT) == kb.KDA_ERR_UNSUPPORTED
        assert call_ex(kern | kb.KDA_FLAG_GATE_SOFTPLUS) == kb.KDA_ERR_UNSUPPORTED
        # a valid kernel passes the flag checks and then meets the (too small) workspace
        assert call_ex(kern) == kb.KDA_ERR_WORKSPACE
    sched = ctypes.c_int32(-1)
    assert lib.kda_fwd_schedule(4, kb.KDA_KERNEL_CHUNK16, ctypes.byref(sched)) == kb.KDA_ERR_INVALID_ARG


def test_binding_refuses_host_tensors():
    import torch
    x = torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kb.kda_fwd(x, x, x, x, torch.zeros(1, 4, 1, dtype=torch.bfloat16), 1.0, x.clone(),
                   torch.zeros(1), torch.zeros(1, 128), -5.0, workspace=torch.zeros(512, dtype=torch.uint8))


def test_host_entry_device_bytes(lib):
    tok = 64 * 2 * 128 * 2
    n = lib.kda_fwd_host_device_bytes(1, 64, 2, 0, -1, -1)
    assert n >= 5 * tok and n % 256 == 0
    assert lib.kda_fwd_host_device_bytes(1, 64, 2, 3, kb.KDA_F32, kb.KDA_F32) >= n + 2 * 3 * 2 * 128 * 128 * 4
    assert lib.kda_fwd_host_device_bytes(-1, 64, 2, 0, -1, -1) == 0
    off = lib.kda_fwd_host_workspace_offset(1, 64, 2, 0, -1, -1)
    assert 5 * tok <= off < n and off % 256 == 0


def test_host_entry_rejects_before_enqueueing(lib):
    """Host-side checks of kda_fwd_host return before any CUDA call: the tensors are host
    descriptors (only cu_seqlens is read, from real host memory) and the device buffer a
    fake aligned address."""
    import numpy as np
    H, Tn = 2, 64
    host = BASE  # never dereferenced except cu_seqlens below

    def run(cu_vals=None, dev=BASE + 0x10000000, nbytes=1 << 40, lb=-5.0):
        cu_arr = None if cu_vals is None else np.asarray(cu_vals, dtype=np.int64)
        cu = None if cu_arr is None else T(kb.KDA_I64, (len(cu_vals),), cu_arr.ctypes.data)
        d = lambda dt, shape: T(dt, shape, host)
        r = lambda x: None if x is None else ctypes.byref(x)
        q = d(kb.KDA_BF16, (1, Tn, H, 128))
        return lib.kda_fwd_host(r(q), r(q), r(q), r(q), r(d(kb.KDA_BF16, (1, Tn, H))), ctypes.c_float(0.1), r(q),
                                r(d(kb.KDA_F32, (H,))), r(d(kb.KDA_F32, (H, 128))), ctypes.c_float(lb), None,
                                None, r(cu), ctypes.c_void_p(dev), ctypes.c_size_t(nbytes), 4, ctypes.c_void_p(0))

    assert run(cu_vals=[1, 10, 64]) == kb.KDA_ERR_INVALID_ARG        # cu_seqlens[0] != 0
    assert run(cu_vals=[0, 40, 30]) == kb.KDA_ERR_INVALID_ARG        # decreasing
    assert run(cu_vals=[0, 40, 65]) == kb.KDA_ERR_INVALID_ARG        # past the tokens
    assert run(nbytes=1024) == kb.KDA_ERR_WORKSPACE                  # device buffer too small
    assert run(dev=BASE + 0x10000000 + 16) == kb.KDA_ERR_WORKSPACE   # misaligned
    assert run(lb=-6.0) == kb.KDA_ERR_UNSUPPORTED                    # the checks of kda_fwd
    assert lib.kda_last_error()


def test_decode_rejects_before_enqueueing(lib):
    B, H = 2, 3
    t = lambda shape, dt=kb.KDA_BF16, off=0: T(dt, shape, BASE + off)

    def call_dec(**over):
        a = dict(q=t((B, H, 128)), k=t((B, H, 128), off=0x100000), v=t((B, H, 128), off=0x200000),
                 g=t((B, H, 128), off=0x300000), beta=t((B, H), off=0x400000), out=t((B, H, 128), off=0x500000),
                 A_log=t((H,), kb.KDA_F32, 0x600000), dt_bias=t((H, 128), kb.KDA_F32, 0x700000), lb=-5.0,
                 init=None, final=None)
        a.update(over)
        r = lambda d: None if d is None else ctypes.byref(d)
        return lib.kda_decode(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]), ctypes.c_float(0.1),
                              r(a["out"]), r(a["A_log"]), r(a["dt_bias"]), ctypes.c_float(a["lb"]), r(a["init"]),
                              r(a["final"]), ctypes.c_void_p(0))

    st4 = lambda dt, off: t((B, H, 128, 128), dt, 0x800000 + off)
    cases = [
        (dict(q=t((B, H, 128, 1))), kb.KDA_ERR_INVALID_ARG),
        (dict(q=t((B, H, 64))), kb.KDA_ERR_UNSUPPORTED),
        (dict(k=t((B, H + 1, 128), off=0x100000)), kb.KDA_ERR_INVALID_ARG),
        (dict(beta=t((B, H, 1), off=0x400000)), kb.KDA_ERR_INVALID_ARG),
        (dict(dt_bias=t((H, 128), kb.KDA_F32, 0x700000 + 4)), kb.KDA_ERR_INVALID_ARG),
        (dict(lb=0.5), kb.KDA_ERR_INVALID_ARG),
        (dict(init=st4(kb.KDA_F32, 0), final=st4(kb.KDA_F32, 4096)), kb.KDA_ERR_ALIAS),
        (dict(init=t((B, H, 128, 64), kb.KDA_F32, 0x800000)), kb.KDA_ERR_INVALID_ARG),
    ]
    for over, expect in cases:
        got = call_dec(**over)
        assert got == expect, (over, got, lib.kda_last_error())


def test_schedule_query_rejects_before_touching_the_device(lib):
    sched = ctypes.c_int32(-1)
    assert lib.kda_fwd_schedule(-1, 0, ctypes.byref(sched)) == kb.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_schedule(8, 0x4, ctypes.byref(sched)) == kb.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_schedule(8, 0, None) == kb.KDA_ERR_INVALID_ARG
    assert sched.value == -1


def test_trace_setter_checks_its_arguments(lib):
    assert lib.kda_fwd_set_trace(ctypes.c_void_p(4), 1024, 0) == kb.KDA_ERR_INVALID_ARG     # misaligned
    assert lib.kda_fwd_set_trace(ctypes.c_void_p(4096), 8, 0) == kb.KDA_ERR_INVALID_ARG    # under one chunk
    assert lib.kda_fwd_set_trace(ctypes.c_void_p(4096), 1024, -1) == kb.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_set_trace(None, 0, 0) == kb.KDA_OK                                  # off


def _header_constants():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    consts = {}
    for name, val in re.findall(r"#define\s+(KDA_[A-Z0-9_]+)\s+\(?(-?0x[0-9a-fA-F]+|-?[0-9.]+)u?f?\)?", text):
        consts[name] = float(val) if "." in val else int(val, 0)
    for name, val in re.findall(r"\b(KDA_[A-Z0-9_]+)\s*=\s*([0-9]+)", text):
        consts[name] = int(val)
    return consts


def test_binding_constants_match_the_header():
    consts = _header_constants()
    mirrored = ["KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED", "KDA_ERR_ALIAS", "KDA_ERR_WORKSPACE",
                "KDA_ERR_CUDA", "KDA_BF16", "KDA_F32", "KDA_I64", "KDA_DEVERR_CU_SEQLENS", "KDA_DEVERR_TIMEOUT",
                "KDA_DEVERR_INTERNAL", "KDA_FLAG_BETA_LOGIT", "KDA_FLAG_GATE_SOFTPLUS", "KDA_FLAG_KERNEL_MASK",
                "KDA_KERNEL_DEFAULT", "KDA_KERNEL_CHUNK16", "KDA_KERNEL_REGISTER_STATE", "KDA_KERNEL_BF16_STATE",
                "KDA_KERNEL_SMEM_STATE",
                "KDA_SCHEDULE_TWO_PER_SM",
                "KDA_SCHEDULE_ONE_PER_SM", "KDA_SCHEDULE_CLUSTER", "KDA_SCHEDULE_CLUSTER2", "KDA_TRACE_POINTS"]
    for name in mirrored:
        assert name in consts, name
        assert getattr(kb, name) == consts[name], name
    assert kb.HEAD_DIM == consts["KDA_HEAD_DIM"]
