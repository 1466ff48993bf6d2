"""The C-ABI library: it builds for sm_103a, loads, exports every function the
header declares, and rejects bad arguments on the host (no GPU needed: the
validation runs before any device call, and no kernel is launched)."""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import pytest

import attention_fa2_fwd_02_gb300 as fa

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def L():
    fa.build()
    return fa.lib()


def _declared_functions():
    text = (ROOT / "include" / "fa.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = _declared_functions()
    assert {"fa_fwd", "fa_fwd_grouped", "fa_check", "fa_status_string", "fa_last_error",
            "fa_debug_set", "fa_version"} <= set(names)


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), f"libfa.so does not export {name}"


def test_library_is_built_for_sm103a():
    # the object files are compiled with exactly one -gencode for sm_103a
    from attention_fa2_fwd_02_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert fa.LIB_PATH.exists()


def test_status_strings(L):
    assert L.fa_status_string(0) == b"ok"
    assert L.fa_status_string(4) == b"device wait timed out"
    assert L.fa_version() == 105


def _t(ptr, strides):
    return fa.FaTensor(ctypes.c_void_p(ptr), (ctypes.c_int64 * 4)(*strides))


def _call(L, dtype=fa.FA_BF16, B=1, H=1, Nq=256, Nk=256, d=128, qptr=0x10000, strides=None,
          scale=0.1, causal=0, lse=None):
    s = strides or (Nq * d, Nq * d, d, 1)
    Q = _t(qptr, s)
    K = _t(0x20000, s)
    V = _t(0x30000, s)
    O = _t(0x40000, s)
    ls = (ctypes.c_int64 * 3)(Nq, Nq, 1)
    return L.fa_fwd(dtype, B, H, Nq, Nk, d, ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V),
                    scale, causal, ctypes.byref(O), lse, ls, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=0), fa.FA_ERR_INVALID_ARG),
    (dict(qptr=0), fa.FA_ERR_INVALID_ARG),
    (dict(strides=(256 * 128, 256 * 128, 128, 2)), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),   # 0, 1 (top-left), 2 (bottom-right)
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
    (dict(d=100), fa.FA_ERR_UNSUPPORTED),   # a row of 200 bytes: not a multiple of 16
    (dict(d=264), fa.FA_ERR_UNSUPPORTED),   # above the 256-column tile
    (dict(d=136, dtype=fa.FA_FP32), fa.FA_ERR_UNSUPPORTED),  # fp32: up to 128
    (dict(qptr=0x10002), fa.FA_ERR_UNSUPPORTED),                     # misaligned base
    (dict(strides=(256 * 128, 256 * 128, 129, 1)), fa.FA_ERR_UNSUPPORTED),  # odd row stride
    (dict(strides=(256 * 128, -128, 128, 1)), fa.FA_ERR_UNSUPPORTED),
])
def test_host_validation(L, kw, status):
    assert _call(L, **kw) == status
    assert L.fa_last_error() != b""


def test_null_tensor_struct(L):
    ls = (ctypes.c_int64 * 3)(1, 1, 1)
    assert L.fa_fwd(0, 1, 1, 1, 1, 128, None, None, None, 1.0, 0, None, None, ls, None) == \
        fa.FA_ERR_INVALID_ARG


def test_grouped_validates_every_problem_first(L):
    good = fa.FaProblem()
    good.B = good.H = 1
    good.N_q = good.N_k = 64
    good.d = 16
    for name in ("Q", "K", "V", "O"):
        setattr(good, name, _t(0x10000, (64 * 16, 64 * 16, 16, 1)))
    good.LSE = None
    good.scale = 0.25
    bad = fa.FaProblem()
    ctypes.pointer(bad)[0] = good
    bad.d = 0
    arr = (fa.FaProblem * 2)(good, bad)
    # the bad second problem is reported before anything is launched
    assert L.fa_fwd_grouped(fa.FA_FP32, 2, arr, None) == fa.FA_ERR_INVALID_ARG
    assert b"problem 1" in L.fa_last_error()
    assert L.fa_fwd_grouped(fa.FA_FP32, 0, None, None) == fa.FA_OK


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64)
    with pytest.raises(ValueError):
        fa.fwd(x, x, x)


def _splitkv(L, n_split=2, ws=0x100000, ws_bytes=1 << 30, d=128, Nq=256):
    s = (Nq * d, Nq * d, d, 1)
    Q, K, V, O = (_t(a, s) for a in (0x10000, 0x20000, 0x30000, 0x40000))
    ls = (ctypes.c_int64 * 3)(Nq, Nq, 1)
    return L.fa_fwd_splitkv(fa.FA_BF16, 1, 1, Nq, Nq, d, ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V),
                            0.1, 0, ctypes.byref(O), None, ls, n_split, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(n_split=0), fa.FA_ERR_INVALID_ARG),
    (dict(n_split=9), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),            # no workspace
    (dict(ws=0x100010), fa.FA_ERR_INVALID_ARG),     # not 256-byte aligned
    (dict(ws_bytes=1024), fa.FA_ERR_INVALID_ARG),   # too small
    (dict(d=16), fa.FA_ERR_UNSUPPORTED),            # small-head path does not split
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
])
def test_splitkv_host_validation(L, kw, status):
    assert _splitkv(L, **kw) == status
    assert L.fa_last_error() != b""


def test_splitkv_workspace_size(L):
    # n_split x rows x (d fp32 + 1 fp32 LSE), each part rounded up to 256 bytes
    rows = 2 * 3 * 100
    want = ((2 * rows * 64 * 4 + 255) // 256) * 256 + ((2 * rows * 4 + 255) // 256) * 256
    assert L.fa_fwd_splitkv_workspace_bytes(2, 3, 100, 64, 2) == want
    assert L.fa_fwd_splitkv_workspace_bytes(2, 3, 100, 64, 1) == 0


def _bwd(L, dtype=fa.FA_BF16, d=128, ws=0x100000, ws_bytes=1 << 30, lse=0x50000, N=256):
    s = (N * d, N * d, d, 1)
    t = [_t(a, s) for a in (0x10000, 0x20000, 0x30000, 0x40000, 0x60000, 0x70000, 0x80000, 0x90000)]
    ls = (ctypes.c_int64 * 3)(N, N, 1)
    return L.fa_bwd(dtype, 1, 1, N, N, d, *(ctypes.byref(x) for x in t[:5]), lse, ls, 0.1, 0,
                    *(ctypes.byref(x) for x in t[5:]), ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=fa.FA_FP32), fa.FA_ERR_UNSUPPORTED),  # bf16 only
    (dict(d=100), fa.FA_ERR_UNSUPPORTED),            # a 200-byte row
    (dict(d=136), fa.FA_ERR_UNSUPPORTED),            # the backward stops at 128
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),             # the forward's LSE is required
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0x100080), fa.FA_ERR_INVALID_ARG),       # not 256-byte aligned
    (dict(ws_bytes=4096), fa.FA_ERR_INVALID_ARG),     # too small
])
def test_bwd_host_validation(L, kw, status):
    assert _bwd(L, **kw) == status
    assert L.fa_last_error() != b""


def test_bwd_workspace_size(L):
    # fp32 dQ accumulator + LSE*log2(e) + delta over N_q rounded up to 128, parts 256-aligned
    rows = 2 * 3 * 256
    want = ((rows * 64 * 4 + 255) // 256) * 256 + 2 * (((rows * 4) + 255) // 256) * 256
    assert L.fa_bwd_workspace_bytes(2, 3, 200, 64) == want
    assert L.fa_bwd_workspace_bytes(0, 3, 200, 64) == 0
    # other head dims take the accumulator of their tile (64 or 128 columns); above 128: none
    assert L.fa_bwd_workspace_bytes(2, 3, 200, 40) == want
    assert L.fa_bwd_workspace_bytes(2, 3, 200, 96) == L.fa_bwd_workspace_bytes(2, 3, 200, 128)
    assert L.fa_bwd_workspace_bytes(2, 3, 200, 256) == 0


def test_gqa_heads_must_divide(L):
    s = (256 * 64, 256 * 64, 64, 1)
    t = [_t(a, s) for a in (0x10000, 0x20000, 0x30000, 0x40000)]
    ls = (ctypes.c_int64 * 3)(256, 256, 1)
    st = L.fa_fwd_gqa(fa.FA_BF16, 1, 6, 4, 256, 256, 64, ctypes.byref(t[0]), ctypes.byref(t[1]),
                      ctypes.byref(t[2]), 0.1, 0, ctypes.byref(t[3]), None, ls, None)
    assert st == fa.FA_ERR_INVALID_ARG and b"H_kv" in L.fa_last_error()
    st = L.fa_fwd_gqa(fa.FA_BF16, 1, 6, 0, 256, 256, 64, ctypes.byref(t[0]), ctypes.byref(t[1]),
                      ctypes.byref(t[2]), 0.1, 0, ctypes.byref(t[3]), None, ls, None)
    assert st == fa.FA_ERR_INVALID_ARG


def _varlen(L, dtype=fa.FA_BF16, B=2, H=4, H_kv=4, total_q=300, total_k=300, max_len=200, d=128,
            cu_q=0x50000, cu_k=0x60000, causal=0):
    sq = (total_q * H * d, d, H * d, 1)  # [total, H, d] packed rows seen as [1, H, total, d]
    sk = (total_k * H_kv * d, d, H_kv * d, 1)
    t = [_t(0x10000, sq), _t(0x20000, sk), _t(0x30000, sk), _t(0x40000, sq)]
    ls = (ctypes.c_int64 * 3)(0, total_q, 1)
    return L.fa_fwd_varlen(dtype, B, H, H_kv, total_q, total_k, max_len, d, 0, ctypes.c_void_p(cu_q),
                           ctypes.c_void_p(cu_k), ctypes.byref(t[0]), ctypes.byref(t[1]), ctypes.byref(t[2]),
                           0.1, causal, ctypes.byref(t[3]), None, ls, None)


@pytest.mark.parametrize("kw,status", [
    (dict(cu_q=0), fa.FA_ERR_INVALID_ARG),           # offsets are required
    (dict(cu_k=0), fa.FA_ERR_INVALID_ARG),
    (dict(max_len=0), fa.FA_ERR_INVALID_ARG),        # max length >= 1
    (dict(max_len=301), fa.FA_ERR_INVALID_ARG),      # ... and <= total_q
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(H_kv=3), fa.FA_ERR_INVALID_ARG),           # K/V heads must divide the query heads
    (dict(dtype=fa.FA_FP32), fa.FA_ERR_UNSUPPORTED),  # bf16 only
    (dict(d=36), fa.FA_ERR_UNSUPPORTED),             # rows of a multiple of 16 bytes only
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),            # head dims up to 128
])
def test_varlen_host_validation(L, kw, status):
    assert _varlen(L, **kw) == status
    assert L.fa_last_error() != b""


def _bwd_dv(L, dtype=fa.FA_BF16, d=128, d_v=64, ws_bytes=1 << 30, N=256):
    sq = (N * d, N * d, d, 1)
    sv = (N * d_v, N * d_v, d_v, 1)
    # Q, K, V, O, dO, then dQ, dK, dV
    t = [_t(a, s) for a, s in zip((0x10000, 0x20000, 0x30000, 0x40000, 0x60000, 0x70000, 0x80000, 0x90000),
                                  (sq, sq, sv, sv, sv, sq, sq, sv))]
    ls = (ctypes.c_int64 * 3)(N, N, 1)
    return L.fa_bwd_dv(dtype, 1, 1, 1, N, N, d, d_v, *(ctypes.byref(x) for x in t[:5]), 0x50000, ls, 0.1, 0,
                       *(ctypes.byref(x) for x in t[5:]), 0x100000, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=fa.FA_FP32), fa.FA_ERR_UNSUPPORTED),      # bf16 only
    (dict(d_v=136), fa.FA_ERR_UNSUPPORTED),              # the backward stops at 128
    (dict(d=256, d_v=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d_v=100), fa.FA_ERR_UNSUPPORTED),              # a 200-byte row
    (dict(ws_bytes=4096), fa.FA_ERR_INVALID_ARG),        # workspace for max(d, d_v) required
])
def test_bwd_dv_host_validation(L, kw, status):
    assert _bwd_dv(L, **kw) == status
    assert L.fa_last_error() != b""


def test_problem_value_dim_validation(L):
    # fa_problem_t.Dv: negative is an argument error; above the tiles, unsupported
    s = (256 * 64, 256 * 64, 64, 1)
    pb = fa.FaProblem()
    pb.B, pb.H, pb.N_q, pb.N_k, pb.d, pb.H_kv = 1, 2, 256, 256, 64, 0
    pb.Q, pb.K, pb.V, pb.O = (_t(a, s) for a in (0x10000, 0x20000, 0x30000, 0x40000))
    pb.LSE = None
    pb.scale, pb.is_causal = 0.125, 0
    pb.Dv = -8
    assert L.fa_fwd_grouped(fa.FA_BF16, 1, ctypes.byref(pb), None) == fa.FA_ERR_INVALID_ARG
    pb.Dv = 264
    assert L.fa_fwd_grouped(fa.FA_BF16, 1, ctypes.byref(pb), None) == fa.FA_ERR_UNSUPPORTED
    pb.Dv = 136
    assert L.fa_fwd_grouped(fa.FA_FP32, 1, ctypes.byref(pb), None) == fa.FA_ERR_UNSUPPORTED  # fp32 stops at 128


def _fwd_ws(L, dtype=fa.FA_FP32, B=1, H=2, H_kv=2, Nq=256, Nk=300, d=128, ws=0x100000, ws_bytes=1 << 30):
    sq, sk = (H * Nq * d, Nq * d, d, 1), (H_kv * Nk * d, Nk * d, d, 1)
    Q, O = _t(0x10000, sq), _t(0x40000, sq)
    K, V = _t(0x20000, sk), _t(0x30000, sk)
    ls = (ctypes.c_int64 * 3)(H * Nq, Nq, 1)
    return L.fa_fwd_ws(dtype, B, H, H_kv, Nq, Nk, d, ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V),
                       0.1, 0, ctypes.byref(O), None, ls, ws, ws_bytes, None)


def test_fwd_ws_bytes(L):
    # fp32 V^T: B * H_kv rows of d, each N_k rounded up to 32 keys, fp32
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 2, 4, 2, 256, 300, 128) == 2 * 2 * 128 * 320 * 4
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 1, 1, 1, 129, 64, 96) == 96 * 64 * 4
    # a V tile read by one query tile only (one query block, one query head per K/V head): none
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 3, 2, 2, 128, 4096, 128) == 0
    # ... but two query heads per K/V head read each V tile twice
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 1, 2, 1, 128, 64, 64) == 64 * 64 * 4
    # bf16, the small-head path and rejected arguments: none
    assert L.fa_fwd_ws_bytes(fa.FA_BF16, 2, 4, 2, 256, 300, 128) == 0
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 1, 1, 1, 4096, 4096, 16) == 0
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 1, 4, 3, 256, 256, 128) == 0   # H_kv does not divide H
    assert L.fa_fwd_ws_bytes(fa.FA_FP32, 1, 1, 1, 256, 256, 136) == 0   # above the fp32 tile


@pytest.mark.parametrize("kw,status", [
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),             # needed, not given
    (dict(ws=0x100040), fa.FA_ERR_INVALID_ARG),      # not 256-byte aligned
    (dict(ws_bytes=128 * 320 * 4 * 2 - 1), fa.FA_ERR_INVALID_ARG),  # one byte short
    (dict(d=102), fa.FA_ERR_UNSUPPORTED),            # usual validation first (408-byte rows)
    (dict(H_kv=3), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_ws_host_validation(L, kw, status):
    assert _fwd_ws(L, **kw) == status
    assert L.fa_last_error() != b""
