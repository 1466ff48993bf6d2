"""fa_fwd_splitkv_noalloc: the split-KV forward on the library's fixed
per-device scratch, for callers that cannot allocate device memory.

It is compared with the allocating entry points (fa_fwd_splitkv with a
caller workspace, and fa_fwd) and with the fp64 oracle, on two calls in a
row, so that the second call runs on scratch the first one left behind (one
pair puts a smaller problem with fewer splits after a larger one, so that
stale partial results from the first call sit past the second call's
layout).  This file collects last, and its tests also pass on their own in a
fresh process (the first call then does the per-device scratch lookup).
"""
from __future__ import annotations

import ctypes
import math
import re
from pathlib import Path

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import qkv

ROOT = Path(__file__).resolve().parent.parent
TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float32: (3e-3, 2e-3)}   # max-abs O, LSE


def test_header_states_the_scratch_size():
    text = (ROOT / "include" / "fa.h").read_text()
    m = re.search(r"#define FA_SPLITKV_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == fa.SPLITKV_NOALLOC_SCRATCH_BYTES


def test_oversize_problem_is_rejected_on_the_host():
    """Rejected before any device call (this runs without a GPU)."""
    fa.build()
    L = fa.lib()
    B, H, N, d, n_split = 1, 64, 8192, 128, 2
    need = L.fa_fwd_splitkv_workspace_bytes(B, H, N, d, n_split)
    assert need > fa.SPLITKV_NOALLOC_SCRATCH_BYTES
    s = (ctypes.c_int64 * 4)(H * N * d, N * d, d, 1)
    t = [fa.FaTensor(ctypes.c_void_p(0x100000 * (i + 1)), s) for i in range(4)]
    ls = (ctypes.c_int64 * 3)(H * N, N, 1)
    st = L.fa_fwd_splitkv_noalloc(fa.FA_BF16, B, H, N, N, d, ctypes.byref(t[0]), ctypes.byref(t[1]),
                                  ctypes.byref(t[2]), 0.1, 0, ctypes.byref(t[3]), None, ls, n_split, None)
    assert st == fa.FA_ERR_UNSUPPORTED
    msg = L.fa_last_error().decode()
    assert str(need) in msg and str(fa.SPLITKV_NOALLOC_SCRATCH_BYTES) in msg


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)


def _case(dtype, B, H, nq, nk, d, causal, seed):
    Q, K, V = (x.cuda() for x in qkv((B, H, nq, d), (B, H, nk, d), seed, dtype))
    return Q, K, V, causal


def _reference(Q, K, V, causal, n_split):
    """The allocating entry points: fa_fwd_splitkv with a workspace from the
    caller, and the unsplit fa_fwd."""
    O_s, L_s = fa.fwd(Q, K, V, is_causal=causal, split_kv=n_split)
    O_1, L_1 = fa.fwd(Q, K, V, is_causal=causal, split_kv=1)
    return (O_s, L_s), (O_1, L_1)


def _close(a, b, dtype, what):
    to, tl = TOL[dtype]
    (Oa, La), (Ob, Lb) = a, b
    eo = float((Oa.float() - Ob.float()).abs().max())
    el = float((La - Lb).abs().max())
    assert math.isfinite(eo) and math.isfinite(el), f"{what}: non-finite"
    assert eo <= to and el <= tl, f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


# pairs of problems run back to back through the no-alloc entry point
PAIRS = [
    # (dtype, B, H, nq, nk, d, causal, n_split)   n_split None = the library's choice
    [(torch.bfloat16, 1, 2, 300, 4096, 128, False, None), (torch.bfloat16, 2, 3, 257, 3000, 64, True, 3)],
    [(torch.float32, 1, 2, 200, 1500, 128, False, 2), (torch.bfloat16, 1, 4, 513, 2048, 128, False, 4)],
    [(torch.bfloat16, 2, 2, 100, 777, 64, False, 5), (torch.bfloat16, 2, 2, 100, 777, 64, False, 5)],
    [(torch.bfloat16, 2, 4, 700, 3000, 128, False, 6), (torch.float32, 1, 2, 150, 1100, 64, True, 2)],
]


def _oracle_rows(Q, K, V, causal, n_rows=64):
    """The oracle on the first and last rows and a seeded sample of the rest
    of every (b, h) slice: (rows, O_ref [B, H, rows, d], LSE_ref [B, H, rows])."""
    import oracle
    nq = Q.shape[2]
    g = torch.Generator().manual_seed(nq)
    rows = sorted(set([0, 1, nq - 1]) | set(torch.randint(0, nq, (n_rows,), generator=g).tolist()))
    Qh, Kh, Vh = (x.cpu() for x in (Q, K, V))
    O_ref = np.empty((Q.shape[0], Q.shape[1], len(rows), V.shape[3]))
    L_ref = np.empty((Q.shape[0], Q.shape[1], len(rows)))
    for b in range(Q.shape[0]):
        for h in range(Q.shape[1]):
            O_ref[b, h], L_ref[b, h] = oracle.attention(Qh[b, h], Kh[b, h], Vh[b, h], 1.0 / math.sqrt(Q.shape[3]),
                                                        causal, rows=rows)
    return rows, O_ref, L_ref


@pytest.mark.gpu
@pytest.mark.parametrize("pair", PAIRS, ids=["auto_then_causal3", "tf32_then_bf16x4", "same_twice",
                                             "large6_then_small_tf32x2"])
def test_two_calls_in_a_row_match_the_allocating_path(pair):
    _gpu()
    runs = []
    for i, (dtype, B, H, nq, nk, d, causal, n_split) in enumerate(pair):
        Q, K, V, causal = _case(dtype, B, H, nq, nk, d, causal, 5000 + 17 * i + nq + nk + d)
        n = n_split or fa.lib().fa_fwd_splitkv_choose(fa.FA_BF16 if dtype == torch.bfloat16 else fa.FA_FP32,
                                                     B, H, nq, nk, d, int(causal))
        if n_split is None:
            assert n > 1, "the library's choice should split this long-key problem"
        O = torch.full(Q.shape, float("nan"), dtype=dtype, device="cuda")
        Lse = torch.full(Q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
        runs.append((Q, K, V, causal, n, O, Lse, dtype, f"call {i}: {dtype} d={d} {nq}x{nk} causal={causal} n_split={n}"))
    # the two no-alloc calls back to back on one stream: the second reuses
    # the scratch the first one wrote
    for Q, K, V, causal, n, O, Lse, *_ in runs:
        fa.fwd_noalloc(Q, K, V, out=O, lse=Lse, is_causal=causal, split_kv=n)
    fa.check()
    for Q, K, V, causal, n, O, Lse, dtype, what in runs:
        ref_split, ref_plain = _reference(Q, K, V, causal, n)
        fa.check()
        _close((O, Lse), ref_split, dtype, what + " vs fa_fwd_splitkv")
        _close((O, Lse), ref_plain, dtype, what + " vs fa_fwd")
        # and against the oracle itself, on sampled rows of every slice
        rows, O_ref, L_ref = _oracle_rows(Q, K, V, causal)
        to, tl = TOL[dtype]
        eo = float(np.abs(O[:, :, rows].float().cpu().numpy() - O_ref).max())
        el = float(np.abs(Lse[:, :, rows].cpu().numpy() - L_ref).max())
        assert eo <= to and el <= tl, f"{what} vs the oracle: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


@pytest.mark.gpu
def test_second_call_allocates_nothing():
    """After the first call (which looks up the scratch), a call leaves
    PyTorch's allocation count unchanged.  (The device's free-memory figure
    is not compared: it covers the whole device, which other processes and
    the driver share.)"""
    _gpu()
    Q, K, V, _ = _case(torch.bfloat16, 1, 2, 300, 4096, 128, False, 6001)
    O = torch.empty_like(Q)
    Lse = torch.empty(Q.shape[:-1], dtype=torch.float32, device="cuda")
    fa.fwd_noalloc(Q, K, V, out=O, lse=Lse, split_kv=2)
    fa.check()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        fa.fwd_noalloc(Q, K, V, out=O, lse=Lse, split_kv=2)
    fa.check()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    ref, _ = _reference(Q, K, V, False, 2)
    _close((O, Lse), ref, torch.bfloat16, "repeated no-alloc call")


@pytest.mark.gpu
def test_python_binding_requires_out():
    _gpu()
    Q, K, V, _ = _case(torch.bfloat16, 1, 1, 64, 64, 64, False, 6002)
    with pytest.raises(ValueError):
        fa.fwd_noalloc(Q, K, V, out=None)
