"""Pins of the fp64 backward oracle (oracle.attention_bwd) to facts outside it.

Each pin takes a candidate backward ``bwd(Q, K, V, dO, scale, causal) ->
(dQ, dK, dV)`` (numpy, one slice [N, d]) and checks it against:
  * finite differences of the forward oracle (itself pinned in
    test_oracle_pins.py) on inputs where the perturbed values are exact in fp32;
  * torch.autograd through the CPU fp64 scaled_dot_product_attention;
  * the closed forms for Q = 0 and for a single key;
  * invariants: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (every row of P
    sums to one, every row of dS to zero).
A plain-numpy restatement with one planted mistake at a time must trip at
least one pin (the same harness as the forward pins).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch


def _grid(shape, seed, step=2.0 ** -8, lim=4.0):
    """Values on a 2^-8 grid in [-4, 4]: x +- 2^-12 and x +- 2^-13 stay exact in fp32."""
    r = np.random.default_rng(seed)
    return (np.round(r.uniform(-lim, lim, shape) / step) * step).astype(np.float32)


def _loss(fwd, Q, K, V, dO, scale, causal):
    O, _ = fwd(Q, K, V, scale, causal)
    return float(np.sum(O * dO.astype(np.float64)))


def pin_finite_differences(bwd, fwd):
    eps = 2.0 ** -12
    for causal in (False, True, 2):
        Q, K, V, dO = _grid((9, 8), 1), _grid((11, 8), 2), _grid((11, 8), 3), _grid((9, 8), 4)
        scale = 0.375
        dQ, dK, dV = bwd(Q, K, V, dO, scale, causal)
        r = np.random.default_rng(5)
        for which, g in ((0, dQ), (1, dK), (2, dV)):
            E = r.choice([-1.0, 1.0], size=[Q, K, V][which].shape).astype(np.float32)
            def central(h):
                args_p = [a + h * E if i == which else a for i, a in enumerate((Q, K, V))]
                args_m = [a - h * E if i == which else a for i, a in enumerate((Q, K, V))]
                return (_loss(fwd, *args_p, dO, scale, causal) - _loss(fwd, *args_m, dO, scale, causal)) / (2 * h)
            # Richardson extrapolation of two exact steps (the eps^2 term cancels)
            num = (4.0 * central(eps / 2) - central(eps)) / 3.0
            ana = float(np.sum(g * E))
            assert abs(num - ana) <= 1e-6 * (1.0 + abs(ana)), (which, causal, num, ana)


def pin_torch_autograd(bwd, fwd):
    r = np.random.default_rng(7)
    for causal, (nq, nk) in ((False, (13, 10)), (True, (13, 10)), (True, (8, 15)), (2, (8, 15)), (2, (10, 10))):
        Q, K, V, dO = (r.standard_normal(s).astype(np.float32) for s in ((nq, 16), (nk, 16), (nk, 16), (nq, 16)))
        dQ, dK, dV = bwd(Q, K, V, dO, 0.21, causal)
        q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
        if causal is not True and causal == 2:
            mask = torch.ones(nq, nk, dtype=torch.bool).tril(diagonal=nk - nq)
        else:
            mask = torch.ones(nq, nk, dtype=torch.bool).tril() if causal else None
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask, scale=0.21)[0]
        (o * torch.tensor(dO, dtype=torch.float64)).sum().backward()
        for got, want in ((dQ, q.grad), (dK, k.grad), (dV, v.grad)):
            np.testing.assert_allclose(got, want.numpy(), rtol=0, atol=1e-12)


def pin_q_zero(bwd, fwd):
    r = np.random.default_rng(11)
    N_q, N_k, d, scale = 6, 5, 4, 0.7
    Q = np.zeros((N_q, d), np.float32)
    K, V = r.standard_normal((N_k, d)).astype(np.float32), r.standard_normal((N_k, d)).astype(np.float32)
    dO = r.standard_normal((N_q, d)).astype(np.float32)
    dQ, dK, dV = bwd(Q, K, V, dO, scale, False)
    Kd, Vd, Gd = K.astype(np.float64), V.astype(np.float64), dO.astype(np.float64)
    # uniform P = 1/N_k: dV_j = mean_i... = sum_i dO_i / N_k; dK = scale dS^T Q = 0;
    # dQ_i = scale / N_k * sum_j (dO_i . (V_j - mean V)) K_j
    np.testing.assert_allclose(dV, np.tile(Gd.sum(0) / N_k, (N_k, 1)), atol=1e-12)
    np.testing.assert_allclose(dK, 0.0, atol=1e-12)
    Vc = Vd - Vd.mean(0)
    np.testing.assert_allclose(dQ, scale / N_k * (Gd @ Vc.T) @ Kd, atol=1e-12)


def pin_single_key(bwd, fwd):
    r = np.random.default_rng(13)
    Q, K, V, dO = (r.standard_normal(s).astype(np.float32) for s in ((7, 8), (1, 8), (1, 8), (7, 8)))
    for causal in (False, True):
        dQ, dK, dV = bwd(Q, K, V, dO, 0.4, causal)
        # P = 1 on the one key: dS = dP - delta = 0, dV_0 = sum_i dO_i
        np.testing.assert_allclose(dQ, 0.0, atol=1e-12)
        np.testing.assert_allclose(dK, 0.0, atol=1e-12)
        np.testing.assert_allclose(dV[0], dO.astype(np.float64).sum(0), atol=1e-12)


def pin_invariants(bwd, fwd):
    r = np.random.default_rng(17)
    for causal in (False, True):
        Q, K, V, dO = (r.standard_normal(s).astype(np.float32) for s in ((12, 8), (12, 8), (12, 8), (12, 8)))
        dQ, dK, dV = bwd(Q, K, V, dO, 0.33, causal)
        np.testing.assert_allclose(dK.sum(0), 0.0, atol=1e-12)
        np.testing.assert_allclose(dV.sum(0), dO.astype(np.float64).sum(0), atol=1e-12)
        assert np.abs(dQ).max() > 1e-3 and np.abs(dK).max() > 1e-3  # not trivially zero


PINS = [pin_finite_differences, pin_torch_autograd, pin_q_zero, pin_single_key, pin_invariants]


@pytest.fixture(scope="module")
def oracle_fns(oracle_mod):
    def bwd(Q, K, V, dO, scale, causal):
        return oracle_mod.attention_bwd(Q, K, V, dO, scale, causal)

    def fwd(Q, K, V, scale, causal):
        return oracle_mod.attention(Q, K, V, scale, causal)
    return bwd, fwd


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_bwd_pin(pin, oracle_fns):
    pin(*oracle_fns)


def test_oracle_bwd_row_subsets_and_batching(oracle_mod):
    r = np.random.default_rng(19)
    Q, dO = r.standard_normal((2, 3, 20, 8)).astype(np.float32), r.standard_normal((2, 3, 20, 8)).astype(np.float32)
    K, V = r.standard_normal((2, 3, 17, 8)).astype(np.float32), r.standard_normal((2, 3, 17, 8)).astype(np.float32)
    for causal in (False, True):
        full = oracle_mod.attention_bwd(Q, K, V, dO, 0.5, causal)
        qr, kr = [19, 0, 7], [16, 3]
        sub = oracle_mod.attention_bwd(Q, K, V, dO, 0.5, causal, q_rows=qr, k_rows=kr)
        np.testing.assert_array_equal(sub[0], full[0][..., qr, :])
        np.testing.assert_array_equal(sub[1], full[1][..., kr, :])
        np.testing.assert_array_equal(sub[2], full[2][..., kr, :])
        one = oracle_mod.attention_bwd(Q[1, 2], K[1, 2], V[1, 2], dO[1, 2], 0.5, causal)
        for a, b in zip(one, full):
            np.testing.assert_array_equal(a, b[1, 2])


# ------------------------------------------------------------------ mutants
def _numpy_bwd(kind):
    """Plain numpy restatement of the backward with one planted mistake."""
    def bwd(Q, K, V, dO, scale, causal):
        Qd, Kd, Vd, Gd = (x.astype(np.float64) for x in (Q, K, V, dO))
        S = scale * Qd @ Kd.T
        if causal:
            k = S.shape[1] - S.shape[0] if (causal is not True and causal == 2) else 0
            S = np.where(np.tri(*S.shape, k=k, dtype=bool), S, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        O = P @ Vd
        dP = Gd @ Vd.T
        delta = (Gd * O).sum(1, keepdims=True)
        dS = P * (dP - delta)
        if kind == "ds_sign":
            dS = -dS
        if kind == "no_delta":
            dS = P * dP
        dV = P.T @ Gd
        if kind == "dv_uses_o":
            dV = P.T @ O
        dQ = scale * dS @ Kd
        if kind == "dq_uses_v":
            dQ = scale * dS @ Vd
        dK = scale * dS.T @ Qd
        if kind == "dk_no_scale":
            dK = dS.T @ Qd
        if kind == "delta_from_v":
            dS = P * (dP - (Gd * Vd.mean(0)).sum(1, keepdims=True))
            dQ, dK = scale * dS @ Kd, scale * dS.T @ Qd
        return dQ, dK, dV
    return bwd


def _numpy_fwd(Q, K, V, scale, causal):
    Qd, Kd, Vd = (x.astype(np.float64) for x in (Q, K, V))
    S = scale * Qd @ Kd.T
    if causal:
        k = S.shape[1] - S.shape[0] if (causal is not True and causal == 2) else 0
        S = np.where(np.tri(*S.shape, k=k, dtype=bool), S, -np.inf)
    m = S.max(1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(1, keepdims=True)
    return (P / l) @ Vd, (m + np.log(l))[:, 0]


MUTANTS = ["ds_sign", "no_delta", "dv_uses_o", "dq_uses_v", "dk_no_scale", "delta_from_v"]


def test_correct_numpy_bwd_passes_all_pins():
    for pin in PINS:
        pin(_numpy_bwd("none"), _numpy_fwd)


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_bwd_mistake_trips_a_pin(kind):
    tripped = []
    for pin in PINS:
        try:
            pin(_numpy_bwd(kind), _numpy_fwd)
        except AssertionError:
            tripped.append(pin.__name__)
    assert tripped, f"mutant {kind} passed every pin"


# ----------------------------------------------------------------------------
# V with a head dim of its own (d_v != d): the same two independent pins
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True, 2])
def test_value_dim_finite_differences(oracle_mod, causal):
    eps = 2.0 ** -12
    Q, K, V, dO = _grid((9, 8), 21), _grid((11, 8), 22), _grid((11, 12), 23), _grid((9, 12), 24)
    scale = 0.375
    dQ, dK, dV = oracle_mod.attention_bwd(Q, K, V, dO, scale, causal)
    assert dQ.shape == (9, 8) and dK.shape == (11, 8) and dV.shape == (11, 12)
    r = np.random.default_rng(25)
    for which, g in ((0, dQ), (1, dK), (2, dV)):
        E = r.choice([-1.0, 1.0], size=[Q, K, V][which].shape).astype(np.float32)

        def central(h):
            args_p = [a + h * E if i == which else a for i, a in enumerate((Q, K, V))]
            args_m = [a - h * E if i == which else a for i, a in enumerate((Q, K, V))]
            return (_loss(oracle_mod.attention, *args_p, dO, scale, causal)
                    - _loss(oracle_mod.attention, *args_m, dO, scale, causal)) / (2 * h)
        num = (4.0 * central(eps / 2) - central(eps)) / 3.0
        ana = float(np.sum(g * E))
        assert abs(num - ana) <= 1e-6 * (1.0 + abs(ana)), (which, causal, num, ana)


@pytest.mark.parametrize("d,d_v", [(16, 24), (24, 8)])
def test_value_dim_torch_autograd(oracle_mod, d, d_v):
    r = np.random.default_rng(26)
    for causal, (nq, nk) in ((False, (13, 10)), (True, (13, 10)), (2, (8, 15))):
        Q, K = r.standard_normal((nq, d)).astype(np.float32), r.standard_normal((nk, d)).astype(np.float32)
        V, dO = r.standard_normal((nk, d_v)).astype(np.float32), r.standard_normal((nq, d_v)).astype(np.float32)
        dQ, dK, dV = oracle_mod.attention_bwd(Q, K, V, dO, 0.3, causal)
        q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (Q, K, V))
        if causal is not True and causal == 2:
            mask = torch.ones(nq, nk, dtype=torch.bool).tril(diagonal=nk - nq)
        else:
            mask = torch.ones(nq, nk, dtype=torch.bool).tril() if causal else None
        o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=mask, scale=0.3)[0]
        (o * torch.tensor(dO, dtype=torch.float64)).sum().backward()
        for got, want in ((dQ, q.grad), (dK, k.grad), (dV, v.grad)):
            np.testing.assert_allclose(got, want.numpy(), rtol=0, atol=1e-12)
