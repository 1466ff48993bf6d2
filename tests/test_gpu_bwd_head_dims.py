"""The backward for head dims other than 64 and 128 and for V with a head dim
of its own (fa_bwd_dv), against the fp64 backward oracle.

The backward kernel's tiles are 64 or 128 columns wide; Q, K (past d) and V,
dO (past d_v) load as zeros and only d / d_v columns of dQ, dK and dV are
stored.  The outputs are views of wider NaN-filled buffers, so a store past
the true head dim fails the test.  Tolerance as in test_gpu_bwd.py:
1.5e-2 * max|ref| + 1e-3 per output tensor."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, qkv

pytestmark = pytest.mark.gpu
RTOL, ATOL = 1.5e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _wide_nan(shape):
    buf = torch.full((*shape[:-1], shape[-1] + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    return buf, buf[..., :shape[-1]]


def _run(oracle_mod, d, dv, causal, B=2, H=3, H_kv=None, nq=300, nk=333, seed=0):
    H_kv = H_kv or H
    Q, K, _ = qkv((B, H, nq, d), (B, H_kv, nk, d), 3000 + seed, torch.bfloat16)
    V = normal((B, H_kv, nk, dv), 3100 + seed, torch.bfloat16)
    G = normal((B, H, nq, dv), 3200 + seed, torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    Qd, Kd, Vd, Gd = Q.cuda(), K.cuda(), V.cuda(), G.cuda()
    O, L = fa.fwd(Qd, Kd, Vd, scale=scale, is_causal=causal)
    bufs = [_wide_nan(x.shape) for x in (Q, K, V)]
    dQ, dK, dV = fa.bwd(Qd, Kd, Vd, O, L, Gd, scale=scale, is_causal=causal,
                        dQ=bufs[0][1], dK=bufs[1][1], dV=bufs[2][1])
    fa.check()
    for name, (buf, _) in zip(("dQ", "dK", "dV"), bufs):
        assert torch.isnan(buf[..., -8:]).all(), f"{name}: a column past the head dim was written"
    G_ = H // H_kv
    rq, rk, rv = oracle_mod.attention_bwd(Q, K.repeat_interleave(G_, 1), V.repeat_interleave(G_, 1), G, scale,
                                          fa.causal_code(causal))
    if G_ > 1:
        rk = rk.reshape(B, H_kv, G_, nk, d).sum(2)
        rv = rv.reshape(B, H_kv, G_, nk, dv).sum(2)
    for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        g = got.float().cpu().numpy()
        assert np.isfinite(g).all(), f"{name} non-finite"
        err = float(np.abs(g - ref).max())
        bound = RTOL * float(np.abs(ref).max()) + ATOL
        assert err <= bound, f"{name}: max|err|={err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("d", [16, 32, 48, 80, 96, 112])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"], ids=["nc", "top_left", "bottom_right"])
def test_bwd_head_dims(oracle_mod, d, causal):
    _run(oracle_mod, d, d, causal, nq=300, nk=333 if causal != "bottom_right" else 200, seed=d)


@pytest.mark.parametrize("d,dv", [(128, 64), (64, 128), (96, 64), (40, 104), (128, 32), (16, 48)])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bwd_value_dim(oracle_mod, d, dv, causal):
    _run(oracle_mod, d, dv, causal, nq=257, nk=385, seed=d + 3 * dv)


@pytest.mark.parametrize("H,H_kv", [(6, 2), (4, 1)])
def test_bwd_value_dim_grouped_heads(oracle_mod, H, H_kv):
    _run(oracle_mod, 128, 64, True, H=H, H_kv=H_kv, nq=300, nk=300, seed=40 + H_kv)
    _run(oracle_mod, 96, 96, False, H=H, H_kv=H_kv, nq=129, nk=500, seed=50 + H_kv)


def test_autograd_and_sdpa_with_value_dim(oracle_mod):
    import torch.nn.functional as F

    from attention_fa2_fwd_02_gb300 import sdpa
    Q, K, _ = qkv((1, 4, 200, 96), (1, 4, 260, 96), 3300, torch.bfloat16)
    V = normal((1, 4, 260, 64), 3301, torch.bfloat16)
    G = normal((1, 4, 200, 64), 3302, torch.bfloat16)
    scale = 1.0 / math.sqrt(96)
    refs = oracle_mod.attention_bwd(Q, K, V, G, scale, True)
    for route in ("attention", "sdpa"):
        q, k, v = (x.cuda().requires_grad_(True) for x in (Q, K, V))
        if route == "attention":
            o = fa.attention(q, k, v, scale=scale, is_causal=True)
        else:
            with sdpa.routed():
                o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        o.backward(G.cuda())
        fa.check()
        for name, got, ref in zip(("dQ", "dK", "dV"), (q.grad, k.grad, v.grad), refs):
            err = float(np.abs(got.float().cpu().numpy() - ref).max())
            assert err <= RTOL * float(np.abs(ref).max()) + ATOL, f"{route} {name}: {err:.3e}"
