"""scaled_dot_product_attention routed to this library (sdpa.py)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300 import sdpa
from attention_fa2_fwd_02_gb300.inputs import normal, qkv


def test_unsupported_arguments_raise():
    x = torch.zeros(1, 1, 8, 64)
    with pytest.raises(NotImplementedError):
        sdpa.scaled_dot_product_attention(x, x, x, attn_mask=torch.ones(8, 8, dtype=torch.bool))
    with pytest.raises(NotImplementedError):
        sdpa.scaled_dot_product_attention(x, x, x, dropout_p=0.1)
    with pytest.raises(ValueError):
        sdpa.scaled_dot_product_attention(torch.zeros(1, 4, 8, 64), x, x)  # GQA needs enable_gqa


def test_routed_restores_the_original():
    orig = F.scaled_dot_product_attention
    with sdpa.routed():
        assert F.scaled_dot_product_attention is sdpa.scaled_dot_product_attention
    assert F.scaled_dot_product_attention is orig
    with pytest.raises(RuntimeError):
        with sdpa.routed():
            raise RuntimeError("inside")
    assert F.scaled_dot_product_attention is orig


gpu = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()


@gpu
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_sdpa_matches_oracle_and_fa(oracle_mod, causal):
    _need_gpu()
    Q, K, V = qkv((2, 4, 300, 128), (2, 4, 300, 128), 1301, torch.bfloat16)
    q, k, v = Q.cuda(), K.cuda(), V.cuda()
    with sdpa.routed():
        o = F.scaled_dot_product_attention(q, k, v, is_causal=causal)
    o2, _ = fa.fwd(q, k, v, is_causal=causal)
    fa.check()
    assert torch.equal(o, o2)
    O_ref, _ = oracle_mod.attention(Q, K, V, 1 / math.sqrt(128), causal)
    assert float(np.abs(o.float().cpu().numpy() - O_ref).max()) <= 2e-2


@gpu
def test_sdpa_autograd_and_gqa(oracle_mod):
    _need_gpu()
    Q, _, _ = qkv((1, 8, 256, 64), (1, 8, 256, 64), 1311, torch.bfloat16)
    _, K, V = qkv((1, 2, 256, 64), (1, 2, 256, 64), 1312, torch.bfloat16)
    dO = normal((1, 8, 256, 64), 1313, torch.bfloat16)
    q, k, v = (x.cuda().requires_grad_(True) for x in (Q, K, V))
    o = sdpa.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True, scale=0.11)
    o.backward(dO.cuda())
    fa.check()
    O, L = fa.fwd(q.detach(), k.detach(), v.detach(), scale=0.11, is_causal=True)
    dQ, dK, dV = fa.bwd(q.detach(), k.detach(), v.detach(), O, L, dO.cuda(), scale=0.11, is_causal=True)
    fa.check()
    assert torch.equal(q.grad, dQ) and torch.equal(k.grad, dK) and torch.equal(v.grad, dV)
    rq, _, _ = oracle_mod.attention_bwd(Q, K.repeat_interleave(4, 1), V.repeat_interleave(4, 1), dO, 0.11, True)
    err = float(np.abs(q.grad.float().cpu().numpy() - rq).max())
    assert err <= 1.5e-2 * float(np.abs(rq).max()) + 1e-3


@gpu
def test_sdpa_inside_torch_compile():
    """The custom op traces as one opaque node (aot_eager backend: no code
    generation), forward and backward."""
    _need_gpu()
    Q, K, V = (x.cuda() for x in qkv((1, 2, 128, 128), (1, 2, 128, 128), 1321, torch.bfloat16))

    def f(q, k, v):
        return sdpa.scaled_dot_product_attention(q, k, v, is_causal=True).float().square().sum()

    cf = torch.compile(f, backend="aot_eager", fullgraph=True)
    q1, k1, v1 = (x.clone().requires_grad_(True) for x in (Q, K, V))
    q2, k2, v2 = (x.clone().requires_grad_(True) for x in (Q, K, V))
    f(q1, k1, v1).backward()
    cf(q2, k2, v2).backward()
    fa.check()
    for a, b in ((q1.grad, q2.grad), (k1.grad, k2.grad), (v1.grad, v2.grad)):
        assert torch.equal(a, b)


@gpu
def test_custom_op_lse_has_no_gradient():
    """The forward custom op returns LSE too, but its backward gives the
    gradients of O only: LSE is marked non-differentiable, so a loss built on
    it cannot silently lose a gradient term."""
    _need_gpu()
    q, k, v = (x.cuda().requires_grad_(True) for x in qkv((1, 2, 128, 64), (1, 2, 128, 64), 1331, torch.bfloat16))
    o, lse = torch.ops.fa_gb300.fwd(q, k, v, 0.125, False)
    fa.check()
    assert o.requires_grad and not lse.requires_grad
    with pytest.raises(RuntimeError):
        lse.sum().backward()
