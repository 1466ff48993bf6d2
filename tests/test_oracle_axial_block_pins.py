"""Pins of the fp64 axial-block oracle (oracle.axial_block): the axial
attention transcript's module (LayerNorm, bias-free QKV projection, 4-head
softmax attention, output projection with bias, residual; row pass then
column pass on the updated grid).

  * PyTorch fp64 on the CPU: nn.LayerNorm / nn.Linear / scaled_dot_product_attention
    assembled as the module's forward;
  * a zero output projection (weight and bias) makes each pass the identity;
  * one-token sequences (W = 1 for the row pass): attention returns the value
    row, so the pass is x + (LN(x) Wv^T) Wo^T + bo in closed form;
  * permuting the W positions permutes the row pass's output the same way
    (attention without positions is permutation-equivariant).
A numpy restatement with one planted mistake at a time trips at least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch


def _params(r, D, scale=0.15):
    return dict(norm_w=1 + 0.1 * r.standard_normal(D), norm_b=0.1 * r.standard_normal(D),
                qkv_w=scale * r.standard_normal((3 * D, D)), out_w=scale * r.standard_normal((D, D)),
                out_b=0.1 * r.standard_normal(D))


def _torch_pass(x, p, heads):
    """The module's _attn_ref + residual with torch layers, fp64 CPU."""
    S, L, D = x.shape
    norm = torch.nn.LayerNorm(D, dtype=torch.float64)
    qkv = torch.nn.Linear(D, 3 * D, bias=False, dtype=torch.float64)
    out = torch.nn.Linear(D, D, dtype=torch.float64)
    with torch.no_grad():
        norm.weight.copy_(torch.from_numpy(np.asarray(p["norm_w"], np.float64)))
        norm.bias.copy_(torch.from_numpy(np.asarray(p["norm_b"], np.float64)))
        qkv.weight.copy_(torch.from_numpy(np.asarray(p["qkv_w"], np.float64)))
        out.weight.copy_(torch.from_numpy(np.asarray(p["out_w"], np.float64)))
        out.bias.copy_(torch.from_numpy(np.asarray(p["out_b"], np.float64)))
        t = qkv(norm(x)).view(S, L, 3, heads, D // heads)
        q, k, v = (t[:, :, i].transpose(1, 2) for i in range(3))
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v).transpose(1, 2).reshape(S, L, D)
        return x + out(o)


def pin_torch_module(block):
    r = np.random.default_rng(1)
    B, H, W, D, heads = 2, 5, 7, 64, 4
    x = r.standard_normal((B, H, W, D))
    row, col = _params(r, D), _params(r, D)
    y = block(x, row, col, heads)
    t = torch.from_numpy(x)
    t = _torch_pass(t.reshape(B * H, W, D), row, heads).reshape(B, H, W, D)
    t = _torch_pass(t.permute(0, 2, 1, 3).reshape(B * W, H, D), col, heads).reshape(B, W, H, D).permute(0, 2, 1, 3)
    np.testing.assert_allclose(y, t.numpy(), rtol=0, atol=1e-12)


def pin_zero_projection_is_identity(block):
    r = np.random.default_rng(2)
    x = r.standard_normal((1, 4, 6, 64))
    zero = _params(r, 64)
    zero["out_w"] = np.zeros((64, 64))
    zero["out_b"] = np.zeros(64)
    np.testing.assert_array_equal(block(x, zero, zero, 4), x)


def pin_single_token_rows(block):
    """W = 1: the row pass is x + (LN(x) Wv^T) Wo^T + bo; the column pass then
    runs on H-long columns (checked against the torch pin's pass)."""
    r = np.random.default_rng(3)
    x = r.standard_normal((2, 3, 1, 64))
    row, col = _params(r, 64), _params(r, 64)
    zero = dict(col, out_w=np.zeros((64, 64)), out_b=np.zeros(64))
    y = block(x, row, zero, 4)                      # column pass = identity
    xd = x.reshape(-1, 64)
    mu = xd.mean(1, keepdims=True)
    ln = (xd - mu) / np.sqrt(((xd - mu) ** 2).mean(1, keepdims=True) + 1e-5) * row["norm_w"] + row["norm_b"]
    v = ln @ row["qkv_w"][128:].T
    want = xd + v @ row["out_w"].T + row["out_b"]
    np.testing.assert_allclose(y.reshape(-1, 64), want, rtol=0, atol=1e-12)


def pin_row_permutation(block):
    r = np.random.default_rng(4)
    x = r.standard_normal((1, 2, 9, 64))
    row = _params(r, 64)
    zero = dict(_params(r, 64), out_w=np.zeros((64, 64)), out_b=np.zeros(64))
    perm = r.permutation(9)
    y = block(x, row, zero, 4)
    yp = block(x[:, :, perm], row, zero, 4)
    np.testing.assert_allclose(yp, y[:, :, perm], rtol=0, atol=1e-12)


PINS = [pin_torch_module, pin_zero_projection_is_identity, pin_single_token_rows, pin_row_permutation]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_axial_block_oracle_pin(pin, oracle_mod):
    pin(oracle_mod.axial_block)


def _numpy_block(kind):
    def ln(x, w, b):
        mu = x.mean(-1, keepdims=True)
        var = ((x - mu) ** 2).mean(-1, keepdims=True)
        if kind == "ln_unbiased_var":
            var = ((x - mu) ** 2).sum(-1, keepdims=True) / (x.shape[-1] - 1)
        return (x - mu) / np.sqrt(var + 1e-5) * w + b

    def one(seqs, p, heads):
        S, L, D = seqs.shape
        d = D // heads
        xn = ln(seqs, p["norm_w"], p["norm_b"])
        qkv = (xn @ p["qkv_w"].T).reshape(S, L, 3, heads, d)
        order = (1, 0, 2) if kind == "q_k_swapped_with_v" else (0, 1, 2)
        q, k, v = (qkv[:, :, i].transpose(0, 2, 1, 3) for i in order)
        sc = q @ k.transpose(0, 1, 3, 2) / (d if kind == "scale_d" else math.sqrt(d))
        pr = np.exp(sc - sc.max(-1, keepdims=True))
        pr /= pr.sum(-1, keepdims=True)
        o = (pr @ v).transpose(0, 2, 1, 3).reshape(S, L, D)
        y = o @ p["out_w"].T + (0 if kind == "no_out_bias" else p["out_b"])
        return y if kind == "no_residual" else seqs + y

    def block(x, row, col, heads):
        B, H, W, D = x.shape
        y = one(x.reshape(B * H, W, D), row, heads).reshape(B, H, W, D)
        src = x if kind == "col_on_input" else y
        yc = one(src.transpose(0, 2, 1, 3).reshape(B * W, H, D), col, heads).reshape(B, W, H, D)
        yc = yc.transpose(0, 2, 1, 3)
        return yc if kind != "col_on_input" else yc + (y - x)
    return block


MUTANTS = ["ln_unbiased_var", "q_k_swapped_with_v", "scale_d", "no_out_bias", "no_residual", "col_on_input"]


def test_numpy_block_passes_all_pins():
    for pin in PINS:
        pin(_numpy_block("none"))


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_block_mistake_trips_a_pin(kind):
    tripped = []
    for pin in PINS:
        try:
            pin(_numpy_block(kind))
        except AssertionError:
            tripped.append(pin.__name__)
    assert tripped, f"mutant {kind} passed every pin"
