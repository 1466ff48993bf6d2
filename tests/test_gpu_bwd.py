"""GPU parity of the backward pass (fa_bwd through the C ABI) against the fp64
backward oracle, on the same seeded inputs.

The GPU backward consumes the GPU forward's own O and LSE, as a training step
does.  Tolerance (max-abs, per output tensor): 1.5e-2 * max|ref| + 1e-3.  The
kernel rounds P and dS to bf16 for the tensor-core products (relative 2^-9
each, in sums over up to N terms), delta uses the bf16 O, and dQ, dK, dV are
stored in bf16 (half an ulp, 2^-9 relative): errors of a few 2^-9 of the
largest magnitude, ~3-6e-3 measured; the bound leaves a factor ~2.5.
"""
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


def _check(name, got, ref, what):
    g = got.float().cpu().numpy() if hasattr(got, "cpu") else got
    assert np.isfinite(g).all(), f"{what}: {name} non-finite"
    err = float(np.abs(g - ref).max())
    bound = RTOL * float(np.abs(ref).max()) + ATOL
    assert err <= bound, f"{what}: {name} max|err|={err:.3e} > {bound:.3e}"


def _run(Q, K, V, G, scale, causal, layout="bhnd"):
    """Host bf16 tensors [B,H,N,d] -> GPU forward + backward -> host grads."""
    if layout == "bnhd":  # head-major storage read and written through strided views
        dev = [x.transpose(1, 2).contiguous().cuda().transpose(1, 2) for x in (Q, K, V, G)]
        outs = [torch.full(x.transpose(1, 2).shape, float("nan"), dtype=x.dtype, device="cuda").transpose(1, 2)
                for x in (Q, K, V)]
    else:
        dev = [x.cuda() for x in (Q, K, V, G)]
        outs = [torch.full(x.shape, float("nan"), dtype=x.dtype, device="cuda") for x in (Q, K, V)]
    Qd, Kd, Vd, Gd = dev
    O, L = fa.fwd(Qd, Kd, Vd, scale=scale, is_causal=causal)
    dQ, dK, dV = fa.bwd(Qd, Kd, Vd, O, L, Gd, scale=scale, is_causal=causal, dQ=outs[0], dK=outs[1], dV=outs[2])
    fa.check()
    return dQ, dK, dV


SHAPES = [(1, 1), (17, 17), (128, 128), (129, 129), (255, 255), (256, 256), (300, 300), (100, 300), (300, 100),
          (257, 1000), (1000, 257), (64, 777)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("nq,nk", SHAPES)
def test_bwd_ragged(oracle_mod, d, causal, nq, nk):
    Q, K, V = qkv((2, 2, nq, d), (2, 2, nk, d), 5000 + 3 * nq + 7 * nk + d, torch.bfloat16)
    G = normal((2, 2, nq, d), 6000 + nq + nk + d, torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    dQ, dK, dV = _run(Q, K, V, G, scale, causal)
    rq, rk, rv = oracle_mod.attention_bwd(Q, K, V, G, scale, causal)
    what = f"d={d} {nq}x{nk} causal={causal}"
    _check("dQ", dQ, rq, what)
    _check("dK", dK, rk, what)
    _check("dV", dV, rv, what)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bwd_strided_head_major(oracle_mod, causal):
    B, H, N, Nk, d = 2, 3, 200, 330, 128
    Q, K, V = qkv((B, H, N, d), (B, H, Nk, d), 71, torch.bfloat16)
    G = normal((B, H, N, d), 72, torch.bfloat16)
    dQ, dK, dV = _run(Q, K, V, G, 0.09, causal, layout="bnhd")
    rq, rk, rv = oracle_mod.attention_bwd(Q, K, V, G, 0.09, causal)
    for n, g, r in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        _check(n, g, r, f"strided causal={causal}")


def test_bwd_causal_keys_no_query_sees(oracle_mod):
    """Causal with N_k > N_q: keys past the last query get exactly zero."""
    Q, K, V = qkv((1, 2, 130, 64), (1, 2, 600, 64), 81, torch.bfloat16)
    G = normal((1, 2, 130, 64), 82, torch.bfloat16)
    dQ, dK, dV = _run(Q, K, V, G, 0.125, True)
    rq, rk, rv = oracle_mod.attention_bwd(Q, K, V, G, 0.125, True)
    assert torch.all(dK[:, :, 130:].float() == 0) and torch.all(dV[:, :, 130:].float() == 0)
    for n, g, r in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        _check(n, g, r, "causal N_k > N_q")


def test_autograd_wrapper_matches_bwd(oracle_mod):
    Q, K, V = qkv((1, 2, 190, 128), (1, 2, 190, 128), 91, torch.bfloat16)
    G = normal((1, 2, 190, 128), 92, torch.bfloat16)
    q, k, v = (x.cuda().requires_grad_(True) for x in (Q, K, V))
    o = fa.attention(q, k, v, is_causal=True)
    o.backward(G.cuda())
    fa.check()
    dQ, dK, dV = _run(Q, K, V, G, 1 / math.sqrt(128), True)
    assert torch.equal(q.grad, dQ) and torch.equal(k.grad, dK) and torch.equal(v.grad, dV)
    rq, rk, rv = oracle_mod.attention_bwd(Q, K, V, G, 1 / math.sqrt(128), True)
    _check("dQ", q.grad, rq, "autograd")


def test_bwd_workspace_reuse_and_repeat():
    """Two calls sharing one workspace give identical results (the dQ
    accumulator is cleared by each call's preprocess)."""
    Q, K, V = (x.cuda() for x in qkv((1, 2, 300, 64), (1, 2, 300, 64), 95, torch.bfloat16))
    G = normal((1, 2, 300, 64), 96, torch.bfloat16).cuda()
    O, L = fa.fwd(Q, K, V)
    ws = torch.empty(fa.lib().fa_bwd_workspace_bytes(1, 2, 300, 64), dtype=torch.uint8, device="cuda")
    a = fa.bwd(Q, K, V, O, L, G, workspace=ws)
    a = [x.clone() for x in a]
    b = fa.bwd(Q, K, V, O, L, G, workspace=ws)
    fa.check()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bwd_full_size_sampled(oracle_mod, causal):
    """B=4 H=32 N=8192 d=128 bf16 (the large self-attention configuration), the
    launch the benchmark times: every output finite; sampled dQ rows and dK,
    dV rows of two (b, h) slices against the oracle."""
    from attention_fa2_fwd_02_gb300.inputs import WORKLOADS
    W = WORKLOADS["large_causal" if causal else "large_nc"]
    Q, K, V = W.make()
    G = normal(Q.shape, 4242, torch.bfloat16)
    Qd, Kd, Vd, Gd = Q.cuda(), K.cuda(), V.cuda(), G.cuda()
    O, L = fa.fwd(Qd, Kd, Vd, scale=W.scale, is_causal=causal)
    dQ, dK, dV = fa.bwd(Qd, Kd, Vd, O, L, Gd, scale=W.scale, is_causal=causal)
    fa.check()
    for t in (dQ, dK, dV):
        assert torch.isfinite(t.float()).all()
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 8191], rng.integers(0, 8192, 26)]))
    for b, h in ((0, 0), (3, 31)):
        rq, rk, rv = oracle_mod.attention_bwd(Q[b, h], K[b, h], V[b, h], G[b, h], W.scale, causal,
                                              q_rows=rows, k_rows=rows)
        what = f"full size b={b} h={h} causal={causal}"
        _check("dQ", dQ[b, h, rows], rq, what)
        _check("dK", dK[b, h, rows], rk, what)
        _check("dV", dV[b, h, rows], rv, what)
