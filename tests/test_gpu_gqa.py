"""Grouped-query attention (K/V with H_kv heads, query head h reading K/V head
h / (H / H_kv)) through fa_fwd_gqa / fa_bwd_gqa, against the oracle applied to
the definition: K and V repeated per query head, and for the backward dK, dV of
a K/V head summed over the query heads that read it."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, qkv

pytestmark = pytest.mark.gpu
FWD_TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float32: (3e-3, 2e-3)}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _expand(x, G):
    return x.repeat_interleave(G, dim=1)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 128),
                                     (torch.float32, 64), (torch.float32, 16), (torch.bfloat16, 32)],
                         ids=["bf16-128", "bf16-64", "fp32-128", "fp32-64", "fp32-16", "bf16-32"])
@pytest.mark.parametrize("H,H_kv", [(6, 1), (6, 2), (6, 3)])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("nq,nk", [(300, 300), (129, 257), (64, 33)])
def test_gqa_forward(oracle_mod, dtype, d, H, H_kv, causal, nq, nk):
    Q, _, _ = qkv((2, H, nq, d), (2, H, nk, d), 700 + nq + d + H_kv, dtype)
    _, K, V = qkv((2, H_kv, nq, d), (2, H_kv, nk, d), 800 + nk + d + H_kv, dtype)
    scale = 1.0 / math.sqrt(d)
    O = torch.full(Q.shape, float("nan"), dtype=dtype, device="cuda")
    L = torch.full(Q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    fa.fwd(Q.cuda(), K.cuda(), V.cuda(), scale=scale, is_causal=causal, out=O, lse=L)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q, _expand(K, H // H_kv), _expand(V, H // H_kv), scale, causal)
    to, tl = FWD_TOL[dtype]
    eo = float(np.abs(O.float().cpu().numpy() - O_ref).max())
    el = float(np.abs(L.cpu().numpy() - L_ref).max())
    assert eo <= to and el <= tl, f"max|dO|={eo:.3e} max|dLSE|={el:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 1), (4, 2)])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("nq,nk", [(300, 300), (200, 333)])
def test_gqa_backward(oracle_mod, d, H, H_kv, causal, nq, nk):
    G = H // H_kv
    Q, _, _ = qkv((2, H, nq, d), (2, H, nk, d), 900 + nq + d, torch.bfloat16)
    _, K, V = qkv((2, H_kv, nq, d), (2, H_kv, nk, d), 950 + nk + d, torch.bfloat16)
    dO = normal((2, H, nq, d), 990 + nq, torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    Qd, Kd, Vd, Gd = Q.cuda(), K.cuda(), V.cuda(), dO.cuda()
    O, L = fa.fwd(Qd, Kd, Vd, scale=scale, is_causal=causal)
    dQ, dK, dV = fa.bwd(Qd, Kd, Vd, O, L, Gd, scale=scale, is_causal=causal)
    fa.check()
    assert dK.shape == K.shape and dV.shape == V.shape
    rq, rk, rv = oracle_mod.attention_bwd(Q, _expand(K, G), _expand(V, G), dO, scale, causal)
    rk = rk.reshape(2, H_kv, G, nk, d).sum(2)
    rv = rv.reshape(2, H_kv, G, nk, d).sum(2)
    for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        g = got.float().cpu().numpy()
        err = float(np.abs(g - ref).max())
        bound = 1.5e-2 * float(np.abs(ref).max()) + 1e-3
        assert np.isfinite(g).all() and err <= bound, f"{name}: max|err|={err:.3e} > {bound:.3e}"


def test_gqa_autograd(oracle_mod):
    Q, _, _ = qkv((1, 8, 256, 128), (1, 8, 256, 128), 1201, torch.bfloat16)
    _, K, V = qkv((1, 2, 256, 128), (1, 2, 256, 128), 1202, torch.bfloat16)
    dO = normal((1, 8, 256, 128), 1203, torch.bfloat16)
    q, k, v = (x.cuda().requires_grad_(True) for x in (Q, K, V))
    fa.attention(q, k, v, is_causal=True).backward(dO.cuda())
    fa.check()
    rq, rk, rv = oracle_mod.attention_bwd(Q, _expand(K, 4), _expand(V, 4), dO, 1 / math.sqrt(128), True)
    rk = rk.reshape(1, 2, 4, 256, 128).sum(2)
    for got, ref in ((q.grad, rq), (k.grad, rk)):
        err = float(np.abs(got.float().cpu().numpy() - ref).max())
        assert err <= 1.5e-2 * float(np.abs(ref).max()) + 1e-3
