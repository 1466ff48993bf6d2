"""Pins of the oracle with a value head dim d_v of its own ("Blackwell
Attention Example", blackwell_attention: Q and K share d, V has Dv columns and
so does O), and with head dims that are not a power of two.

* The columns of O are the softmax weights applied to the matching columns of
  V, so attention(Q, K, [V1 | V2]) = [attention(Q, K, V1) | attention(Q, K, V2)]
  with one LSE: this ties any d_v to the d_v = d case pinned elsewhere.
* V = the identity (d_v = N_k) makes O the softmax weights themselves, which a
  dense numpy softmax gives independently; V = ones (d_v = 1) gives O = 1.
* Brute force against a dense numpy evaluation on tiny inputs for
  d, d_v in {8, 24, 40, 96, 136} and all three causal modes.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle


def _dense(Q, K, V, scale, causal):
    Q, K, V = (x.astype(np.float64) for x in (Q, K, V))
    S = scale * Q @ K.T
    Nq, Nk = S.shape
    i, j = np.arange(Nq)[:, None], np.arange(Nk)[None, :]
    if causal == 1:
        S = np.where(j <= i, S, -np.inf)
    elif causal == 2:
        S = np.where(j <= i + Nk - Nq, S, -np.inf)
    empty = np.isneginf(S).all(1)
    S = np.where(empty[:, None], 0.0, S)
    m = S.max(1, keepdims=True)
    P = np.exp(S - m) * ~np.isneginf(np.where(empty[:, None], -np.inf, S))
    l = P.sum(1)
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(empty[:, None], 0.0, P @ V / l[:, None])
        L = np.where(empty, -np.inf, m[:, 0] + np.log(l))
    return O, L


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_value_columns_split(causal):
    Q, K = _rand((2, 37, 64), 1), _rand((2, 45, 64), 2)
    V1, V2 = _rand((2, 45, 64), 3), _rand((2, 45, 24), 4)
    O, L = oracle.attention(Q, K, np.concatenate([V1, V2], -1), 0.125, causal)
    O1, L1 = oracle.attention(Q, K, V1, 0.125, causal)
    O2, L2 = oracle.attention(Q, K, V2, 0.125, causal)
    assert O.shape == (2, 37, 88)
    np.testing.assert_array_equal(O[..., :64], O1)
    np.testing.assert_array_equal(O[..., 64:], O2)
    np.testing.assert_array_equal(L, L1)
    np.testing.assert_array_equal(L, L2)


@pytest.mark.parametrize("causal", [0, 1])
def test_identity_values_give_the_weights(causal):
    Q, K = _rand((19, 40), 5), _rand((23, 40), 6)
    O, L = oracle.attention(Q, K, np.eye(23, dtype=np.float32), 0.2, causal)
    S = 0.2 * Q.astype(np.float64) @ K.astype(np.float64).T
    if causal:
        S = np.where(np.arange(23)[None, :] <= np.arange(19)[:, None], S, -np.inf)
    P = np.exp(S - S.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    np.testing.assert_allclose(O, P, rtol=0, atol=1e-14)
    assert np.all(O.sum(1) > 1 - 1e-12)


def test_ones_values_give_one():
    Q, K = _rand((3, 30, 96), 7), _rand((3, 50, 96), 8)
    O, _ = oracle.attention(Q, K, np.ones((3, 50, 1), np.float32), 0.1, 0)
    np.testing.assert_allclose(O, 1.0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("d,d_v", [(8, 8), (24, 40), (40, 24), (96, 96), (96, 64), (136, 8), (64, 128)])
@pytest.mark.parametrize("causal", [0, 1, 2])
def test_brute_force(d, d_v, causal):
    Q, K, V = _rand((21, d), 10 + d), _rand((17, d), 11 + d_v), _rand((17, d_v), 12 + d + d_v)
    O, L = oracle.attention(Q, K, V, 1.0 / np.sqrt(d), causal)
    Ob, Lb = _dense(Q, K, V, 1.0 / np.sqrt(d), causal)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    fin = np.isfinite(Lb)
    assert np.array_equal(np.isfinite(L), fin)
    np.testing.assert_allclose(L[fin], Lb[fin], rtol=0, atol=1e-12)


def test_shape_checks():
    Q, K = _rand((5, 16), 20), _rand((6, 16), 21)
    with pytest.raises(ValueError):
        oracle.attention(Q, K, _rand((7, 16), 22), 1.0)   # V rows must match K rows
    with pytest.raises(ValueError):
        oracle.attention(Q, _rand((6, 8), 23), _rand((6, 16), 24), 1.0)  # Q and K share d
