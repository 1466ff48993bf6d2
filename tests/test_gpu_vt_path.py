"""fp32 inputs: the two ways the tf32 P.V gets its K-major V^T operand, both
against the fp64 oracle on the same seeded inputs (O <= 3e-3, LSE <= 2e-3).

  * fa_fwd_ws: fa_vt_kernel writes V^T once into the caller's workspace and
    the attention kernel loads V^T tiles by TMA;
  * fa_fwd_gqa (no workspace): the attention kernel transposes every V tile
    in shared memory.

Covered: ragged N_q / N_k (key counts that are not multiples of the 32-key
V^T block or the 128-key tile), head dims below the tile width (V^T rows past
Dv read as zeros), grouped K/V heads, strided and heads-major V, both causal
alignments (bottom-right with rows that see no key), and a workspace that
holds NaN or an earlier problem's V^T (every value read is written first).
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, qkv

pytestmark = pytest.mark.gpu

TO, TL = 3e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _setup(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _ws_bytes(Q, K, V):
    L = fa.lib()
    q4, k4 = fa._as4(Q), fa._as4(K)
    return L.fa_fwd_ws_bytes(fa.FA_FP32, q4.shape[0], q4.shape[1], k4.shape[1], q4.shape[2], k4.shape[2],
                             q4.shape[3])


def _run(Q, K, V, scale, causal, workspace):
    """One call: with `workspace` (a CUDA uint8 tensor) through fa_fwd_ws, else
    through fa_fwd_gqa.  Outputs start as NaN."""
    O = torch.full(Q.shape[:-1] + (V.shape[-1],), float("nan"), dtype=Q.dtype, device="cuda")
    LSE = torch.full(Q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    pb, O, LSE = fa._problem(Q, K, V, scale, causal, O, LSE, True)
    L = fa.lib()
    ls = (ctypes.c_int64 * 3)(*pb.lse_stride)
    args = (fa.FA_FP32, pb.B, pb.H, pb.H_kv, pb.N_q, pb.N_k, pb.d, ctypes.byref(pb.Q), ctypes.byref(pb.K),
            ctypes.byref(pb.V), pb.scale, pb.is_causal, ctypes.byref(pb.O), pb.LSE, ls)
    stream = fa._stream_ptr(Q.device)
    if workspace is None:
        st = L.fa_fwd_gqa(*args, stream)
    else:
        st = L.fa_fwd_ws(*args, ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), stream)
    fa._raise_on(st)
    fa.check()
    return O.cpu().numpy(), LSE.cpu().numpy()


def _check(O, L, O_ref, L_ref, what):
    fin = np.isfinite(L_ref)
    assert np.isfinite(O).all(), f"{what}: non-finite O"
    assert np.array_equal(np.isfinite(L), fin), f"{what}: LSE finiteness differs"
    eo = float(np.abs(O - O_ref).max())
    el = float(np.abs(L[fin] - L_ref[fin]).max()) if fin.any() else 0.0
    assert eo <= TO and el <= TL, f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


def _oracle(oracle_mod, Q, K, V, scale, causal):
    """The oracle on K/V repeated to the query heads (head h reads K/V head
    h / (H / H_kv)), with the library's causal code (0, 1 top-left, 2 bottom-right)."""
    g = Q.shape[1] // K.shape[1]
    K, V = K.cpu().repeat_interleave(g, dim=1), V.cpu().repeat_interleave(g, dim=1)
    return oracle_mod.attention(Q.cpu(), K, V, scale, fa.causal_code(causal))


def _both(oracle_mod, Q, K, V, scale, causal, what):
    """Both paths against the oracle; the workspace starts as NaN."""
    need = _ws_bytes(Q, K, V)
    assert need > 0, f"{what}: expected the V^T path"
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)
    O_ref, L_ref = _oracle(oracle_mod, Q, K, V, scale, causal)
    Ow, Lw = _run(Q, K, V, scale, causal, ws)
    _check(Ow, Lw, O_ref, L_ref, what + " [V^T pass]")
    Ok, Lk = _run(Q, K, V, scale, causal, None)
    _check(Ok, Lk, O_ref, L_ref, what + " [in-kernel transpose]")


# (B, H, H_kv, N_q, N_k, d, causal)
CASES = [
    (1, 2, 2, 256, 512, 128, False),
    (2, 3, 3, 300, 1000, 64, True),
    (1, 2, 2, 129, 33, 128, False),      # one partial key tile of 33 keys
    (1, 1, 1, 640, 131, 128, True),      # keys past a 32-key block boundary
    (1, 4, 2, 200, 777, 96, False),      # d below the 128-column tile, grouped K/V heads
    (2, 2, 1, 130, 260, 40, True),       # d = 40 on the 64-column tile
    (1, 3, 3, 1000, 1000, 128, True),
    (1, 2, 2, 512, 4096, 64, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}kv{c[2]}_{c[3]}x{c[4]}_d{c[5]}_{'causal' if c[6] else 'nc'}"
                                             for c in CASES])
def test_vt_pass_and_in_kernel_transpose(oracle_mod, case):
    B, H, H_kv, nq, nk, d, causal = case
    Q, K, V = qkv((B, H, nq, d), (B, H_kv, nk, d), 4000 + nq + 3 * nk + d, torch.float32)
    _both(oracle_mod, Q.cuda(), K.cuda(), V.cuda(), 1 / math.sqrt(d), causal, str(case))


def test_bottom_right_rows_without_keys(oracle_mod):
    # N_q > N_k, bottom-right: the first N_q - N_k rows see no key (O = 0, LSE = -inf)
    Q, K, V = qkv((1, 2, 400, 128), (1, 2, 150, 128), 4101, torch.float32)
    _both(oracle_mod, Q.cuda(), K.cuda(), V.cuda(), 1 / math.sqrt(128), "bottom_right", "bottom-right 400x150")


def test_strided_and_heads_major_v(oracle_mod):
    d = 128
    Q, K, _ = qkv((2, 2, 384, d), (2, 2, 500, d), 4202, torch.float32)
    # V with padded rows (row stride d + 4) and V stored [B, N, H, d] (heads-major), viewed as [B, H, N, d]
    big = normal((2, 2, 500, d + 4), 4203)
    V1 = big.cuda()[..., :d]
    V2 = normal((2, 500, 2, d), 4204).cuda().transpose(1, 2)
    for V, what in ((V1, "padded rows"), (V2, "heads-major")):
        assert not V.is_contiguous()
        _both(oracle_mod, Q.cuda(), K.cuda(), V, 1 / math.sqrt(d), False, what)


def test_workspace_reuse_larger_then_smaller(oracle_mod):
    # the second problem's workspace holds the first one's V^T (other N_k, d)
    Q1, K1, V1 = qkv((1, 2, 300, 128), (1, 2, 2000, 128), 4301, torch.float32)
    Q2, K2, V2 = qkv((2, 1, 260, 64), (2, 1, 70, 64), 4302, torch.float32)
    need1 = _ws_bytes(Q1, K1, V1)
    assert need1 > _ws_bytes(Q2, K2, V2) > 0
    ws = torch.empty(need1, dtype=torch.uint8, device="cuda")
    for (Q, K, V), causal in (((Q1, K1, V1), False), ((Q2, K2, V2), True)):
        d = Q.shape[-1]
        O_ref, L_ref = _oracle(oracle_mod, Q, K, V, 1 / math.sqrt(d), causal)
        O, L = _run(Q.cuda(), K.cuda(), V.cuda(), 1 / math.sqrt(d), causal, ws)
        _check(O, L, O_ref, L_ref, f"reuse d={d}")


def test_binding_takes_the_vt_pass_and_accepts_a_workspace(oracle_mod):
    Q, K, V = qkv((1, 2, 256, 128), (1, 2, 256, 128), 4401, torch.float32)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    need = _ws_bytes(Qd, Kd, Vd)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, 1 / math.sqrt(128), False)
    O, L = fa.fwd(Qd, Kd, Vd, split_kv=1)  # workspace from PyTorch's allocator
    _check(O.cpu().numpy(), L.cpu().numpy(), O_ref, L_ref, "binding, own workspace")
    O, L = fa.fwd(Qd, Kd, Vd, split_kv=1, workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
    _check(O.cpu().numpy(), L.cpu().numpy(), O_ref, L_ref, "binding, given workspace")
    with pytest.raises(ValueError):
        fa.fwd(Qd, Kd, Vd, split_kv=1, workspace=torch.empty(need - 1, dtype=torch.uint8, device="cuda"))
