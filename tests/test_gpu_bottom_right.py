"""Bottom-right causal alignment (is_causal = 2: key j visible to query row i
iff j <= i + N_k - N_q) on every path, against the oracle: forward (tensor
core bf16/tf32, split-KV, small-head) and backward.  With N_q > N_k the first
N_q - N_k rows see no key: O = 0, LSE = -inf, zero gradients."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, qkv

pytestmark = pytest.mark.gpu
TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float32: (3e-3, 2e-3)}
SHAPES = [(100, 300), (256, 1000), (300, 300), (513, 200), (1000, 257), (17, 1), (64, 33)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _check_fwd(O, L, O_ref, L_ref, dtype, what):
    O, L = O.float().cpu().numpy(), L.cpu().numpy()
    empty = np.isneginf(L_ref)
    assert np.all(np.isneginf(L[empty])) and np.all(O[empty] == 0), f"{what}: rows that see no key"
    assert np.isfinite(O).all() and np.isfinite(L[~empty]).all(), f"{what}: non-finite"
    to, tl = TOL[dtype]
    eo = float(np.abs(O - O_ref).max())
    el = float(np.abs(L[~empty] - L_ref[~empty]).max()) if (~empty).any() else 0.0
    assert eo <= to and el <= tl, f"{what}: max|dO|={eo:.3e} max|dLSE|={el:.3e}"


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 128),
                                     (torch.float32, 64), (torch.float32, 16), (torch.bfloat16, 32)],
                         ids=["bf16-128", "bf16-64", "fp32-128", "fp32-64", "fp32-16", "bf16-32"])
@pytest.mark.parametrize("nq,nk", SHAPES)
def test_bottom_right_forward(oracle_mod, dtype, d, nq, nk):
    if d <= 32 and nk > 1024:
        pytest.skip("small-head path takes N_k <= 1024")
    Q, K, V = qkv((2, 3, nq, d), (2, 3, nk, d), 1500 + nq + nk + d, dtype)
    scale = 1.0 / math.sqrt(d)
    O = torch.full(Q.shape, float("nan"), dtype=dtype, device="cuda")
    L = torch.full(Q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    fa.fwd(Q.cuda(), K.cuda(), V.cuda(), scale=scale, is_causal="bottom_right", out=O, lse=L, split_kv=1)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, 2)
    _check_fwd(O, L, O_ref, L_ref, dtype, f"{dtype} d={d} {nq}x{nk}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq,nk,split", [(100, 3000, 3), (300, 1000, 2), (700, 300, 2)])
def test_bottom_right_split_kv(oracle_mod, d, nq, nk, split):
    Q, K, V = qkv((1, 2, nq, d), (1, 2, nk, d), 1600 + nq + d, torch.bfloat16)
    O = torch.full(Q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    L = torch.full(Q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    fa.fwd(Q.cuda(), K.cuda(), V.cuda(), scale=0.1, is_causal="bottom_right", out=O, lse=L, split_kv=split)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q, K, V, 0.1, 2)
    _check_fwd(O, L, O_ref, L_ref, torch.bfloat16, f"split={split} d={d} {nq}x{nk}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq,nk", [(100, 300), (300, 300), (513, 200), (200, 777)])
def test_bottom_right_backward(oracle_mod, d, nq, nk):
    Q, K, V = qkv((2, 2, nq, d), (2, 2, nk, d), 1700 + nq + nk + d, torch.bfloat16)
    dO = normal((2, 2, nq, d), 1800 + nq, torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    Qd, Kd, Vd, Gd = Q.cuda(), K.cuda(), V.cuda(), dO.cuda()
    O, L = fa.fwd(Qd, Kd, Vd, scale=scale, is_causal="bottom_right")
    dQ, dK, dV = fa.bwd(Qd, Kd, Vd, O, L, Gd, scale=scale, is_causal="bottom_right")
    fa.check()
    rq, rk, rv = oracle_mod.attention_bwd(Q, K, V, dO, scale, 2)
    for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        g = got.float().cpu().numpy()
        err = float(np.abs(g - ref).max())
        bound = 1.5e-2 * float(np.abs(ref).max()) + 1e-3
        assert np.isfinite(g).all() and err <= bound, f"{name} {nq}x{nk} d={d}: {err:.3e} > {bound:.3e}"


def test_top_left_is_unchanged_by_the_alignment_code(oracle_mod):
    """N_q == N_k: bottom-right equals top-left, bit for bit."""
    Q, K, V = (x.cuda() for x in qkv((1, 2, 300, 128), (1, 2, 300, 128), 1901, torch.bfloat16))
    a, la = fa.fwd(Q, K, V, is_causal=True)
    b, lb = fa.fwd(Q, K, V, is_causal="bottom_right")
    fa.check()
    assert torch.equal(a, b) and torch.equal(la, lb)
