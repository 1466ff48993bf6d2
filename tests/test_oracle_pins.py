"""Pins of the fp64 CPU oracle to facts fixed by the pages and by mathematics.

None of these re-types the oracle's formula or re-calls its routine: each pin
is a closed form, an invariant, an independent formulation (the tiled
online-softmax of "Extend Thunder with CUDA-Python", flash_attention_reference,
written afresh here), or a library routine (PyTorch SDPA on the CPU in fp64).

Every ``pin_*`` takes an attention callable ``attn(Q, K, V, scale, causal)``
returning (O, LSE) as float64 arrays, so that the last test can feed it
deliberately broken variants and show that each one trips at least one pin.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(shape, seed, dtype=np.float32):
    return _rng(seed).standard_normal(shape).astype(dtype)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_q_zero(attn):
    """Q = 0: every score is 0, so O is the mean of the visible V rows and
    LSE = log(#visible)."""
    for (Nq, Nk) in [(5, 9), (9, 5), (6, 6)]:
        d = 4
        Q = np.zeros((Nq, d), np.float32)
        K = _rand((Nk, d), 1)
        V = _rand((Nk, d), 2)
        O, L = attn(Q, K, V, 0.7, False)
        np.testing.assert_allclose(O, np.broadcast_to(V.astype(np.float64).mean(0), O.shape),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(L, np.full(Nq, math.log(Nk)), rtol=0, atol=1e-12)
        O, L = attn(Q, K, V, 0.7, True)
        for i in range(Nq):
            nv = min(i + 1, Nk)
            np.testing.assert_allclose(O[i], V[:nv].astype(np.float64).mean(0), rtol=0, atol=1e-12)
            assert abs(L[i] - math.log(nv)) <= 1e-12


def pin_scale_zero(attn):
    """scale = 0 gives the same closed forms as Q = 0."""
    Q, K, V = _rand((7, 8), 3), _rand((11, 8), 4), _rand((11, 8), 5)
    O, L = attn(Q, K, V, 0.0, False)
    np.testing.assert_allclose(O, np.broadcast_to(V.astype(np.float64).mean(0), O.shape),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, np.full(7, math.log(11)), rtol=0, atol=1e-12)


def pin_single_key(attn):
    """N_k = 1: the softmax weight is 1, O = V[0], LSE = scale * Q_i . K_0."""
    Q, K, V = _rand((6, 5), 6), _rand((1, 5), 7), _rand((1, 5), 8)
    for causal in (False, True):
        O, L = attn(Q, K, V, 0.3, causal)
        np.testing.assert_allclose(O, np.broadcast_to(V[0].astype(np.float64), O.shape),
                                   rtol=0, atol=1e-12)
        want = 0.3 * (Q.astype(np.float64) @ K[0].astype(np.float64))
        np.testing.assert_allclose(L, want, rtol=0, atol=1e-12)


def pin_first_causal_row(attn):
    """Causal, top-left: query row 0 sees key 0 alone, so O[0] = V[0] and
    LSE[0] = scale * Q_0 . K_0, whether N_k is above or below N_q."""
    for (Nq, Nk) in [(8, 8), (4, 10), (10, 4)]:
        Q, K, V = _rand((Nq, 6), 9), _rand((Nk, 6), 10), _rand((Nk, 6), 11)
        O, L = attn(Q, K, V, 0.45, True)
        np.testing.assert_allclose(O[0], V[0].astype(np.float64), rtol=0, atol=1e-12)
        want = 0.45 * float(Q[0].astype(np.float64) @ K[0].astype(np.float64))
        assert abs(L[0] - want) <= 1e-12


def pin_permutation(attn):
    """Non-causal O and LSE do not change under a joint permutation of the
    K and V rows (the softmax sums over keys)."""
    Q, K, V = _rand((9, 7), 12), _rand((13, 7), 13), _rand((13, 7), 14)
    perm = _rng(15).permutation(13)
    O1, L1 = attn(Q, K, V, 0.5, False)
    O2, L2 = attn(Q, K[perm], V[perm], 0.5, False)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-12)
    # and a non-trivial dependence on K: permuting K alone changes the result
    O3, _ = attn(Q, K[perm], V, 0.5, False)
    assert np.abs(O3 - O1).max() > 1e-3


def pin_large_scores(attn):
    """Two keys with scores +x and -x, x = 800 (exp(800) overflows fp64):
    LSE = x + log(1 + e^{-2x}) = x and O = V[0] exactly (weight sigma(2x))."""
    Q = np.array([[2.0]], np.float32)
    K = np.array([[1.0], [-1.0]], np.float32)
    V = np.array([[3.0], [-5.0]], np.float32)
    O, L = attn(Q, K, V, 400.0, False)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    assert abs(O[0, 0] - 3.0) <= 1e-12
    assert abs(L[0] - 800.0) <= 1e-12
    # moderate x keeps both terms: x = 0.5 -> closed form
    O, L = attn(Q, K, V, 0.25, False)
    x = 0.5
    w0 = 1.0 / (1.0 + math.exp(-2 * x))
    assert abs(O[0, 0] - (3.0 * w0 - 5.0 * (1 - w0))) <= 1e-12
    assert abs(L[0] - math.log(math.exp(x) + math.exp(-x))) <= 1e-12


def _online_softmax_tiled(Q, K, V, scale, causal, B_r, B_c):
    """Block-tiled online softmax in fp64, the structure of the tutorial's
    flash_attention_reference (row tiles of B_r, key tiles of B_c, running
    max m, running sum l, rescale by exp(m_old - m_new)), written afresh."""
    Q = Q.astype(np.float64)
    K = K.astype(np.float64)
    V = V.astype(np.float64)
    Nq, d = Q.shape
    Nk = K.shape[0]
    O = np.zeros((Nq, d))
    L = np.zeros(Nq)
    for i0 in range(0, Nq, B_r):
        rows = np.arange(i0, min(i0 + B_r, Nq))
        m = np.full(len(rows), -np.inf)
        l = np.zeros(len(rows))
        acc = np.zeros((len(rows), d))
        for j0 in range(0, Nk, B_c):
            cols = np.arange(j0, min(j0 + B_c, Nk))
            if causal and cols[0] > rows[-1]:
                break
            S = scale * (Q[rows] @ K[cols].T)
            if causal:
                S = np.where(rows[:, None] >= cols[None, :], S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))
            P = np.exp(S - m_new[:, None])
            corr = np.exp(m - m_new)
            l = corr * l + P.sum(axis=1)
            acc = corr[:, None] * acc + P @ V[cols]
            m = m_new
        O[rows] = acc / l[:, None]
        L[rows] = m + np.log(l)
    return O, L


def pin_online_softmax_recompute(attn):
    """The tiled online-softmax recomputation agrees to 1e-12 on tiny inputs,
    tile sizes 16/16 and 7/5, square and rectangular, causal or not."""
    for (Nq, Nk, d, seed) in [(33, 33, 8, 20), (21, 40, 5, 21), (40, 19, 6, 22)]:
        Q, K, V = _rand((Nq, d), seed), _rand((Nk, d), seed + 100), _rand((Nk, d), seed + 200)
        for causal in (False, True):
            O, L = attn(Q, K, V, 0.37, causal)
            for (br, bc) in [(16, 16), (7, 5)]:
                O2, L2 = _online_softmax_tiled(Q, K, V, 0.37, causal, br, bc)
                np.testing.assert_allclose(O, O2, rtol=0, atol=1e-12)
                np.testing.assert_allclose(L, L2, rtol=0, atol=1e-12)


def pin_torch_sdpa(attn):
    """PyTorch SDPA (CPU, float64) and torch.logsumexp of explicit scores agree
    to 1e-12; torch's is_causal is the top-left mask used here."""
    for (Nq, Nk, d, seed) in [(17, 17, 16, 30), (12, 29, 8, 31), (29, 12, 8, 32)]:
        Q, K, V = _rand((Nq, d), seed), _rand((Nk, d), seed + 1), _rand((Nk, d), seed + 2)
        for causal in (False, True):
            O, L = attn(Q, K, V, 0.21, causal)
            tq, tk, tv = (torch.from_numpy(x.astype(np.float64)) for x in (Q, K, V))
            ref = torch.nn.functional.scaled_dot_product_attention(
                tq[None], tk[None], tv[None], is_causal=causal, scale=0.21)[0]
            S = 0.21 * tq @ tk.T
            if causal:
                S = S.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).tril().logical_not(),
                                  float("-inf"))
            lse = torch.logsumexp(S, dim=-1)
            np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(L, lse.numpy(), rtol=0, atol=1e-12)


def pin_invariants(attn):
    """Convex hull of V rows; max s <= LSE <= max s + log(#visible);
    sum_j exp(s_j - LSE) = 1."""
    Q, K, V = _rand((14, 9), 40), _rand((23, 9), 41), _rand((23, 9), 42)
    for causal in (False, True):
        O, L = attn(Q, K, V, 0.6, causal)
        S = 0.6 * (Q.astype(np.float64) @ K.astype(np.float64).T)
        for i in range(14):
            nv = min(i + 1, 23) if causal else 23
            s = S[i, :nv]
            vmin, vmax = V[:nv].min(0), V[:nv].max(0)
            assert np.all(O[i] >= vmin - 1e-12) and np.all(O[i] <= vmax + 1e-12)
            assert s.max() - 1e-12 <= L[i] <= s.max() + math.log(nv) + 1e-12
            assert abs(np.exp(s - L[i]).sum() - 1.0) <= 1e-12


def pin_worked_examples(attn):
    """Hand-derived closed forms stored in tests/golden/worked_examples.json."""
    data = json.loads((GOLDEN / "worked_examples.json").read_text())
    env = {"e": math.e, "exp": math.exp, "log": math.log, "sqrt": math.sqrt}
    for case in data["cases"]:
        Q = np.array(case["Q"], np.float32)
        K = np.array(case["K"], np.float32)
        V = np.array(case["V"], np.float32)
        O, L = attn(Q, K, V, case["scale"], case["causal"])
        O_want = np.array([[eval(x, env) for x in row] for row in case["O"]])
        L_want = np.array([eval(x, env) for x in case["LSE"]])
        np.testing.assert_allclose(O, O_want, rtol=0, atol=1e-12, err_msg=case["name"])
        np.testing.assert_allclose(L, L_want, rtol=0, atol=1e-12, err_msg=case["name"])


def pin_bottom_right_causal(attn):
    """is_causal = 2 (bottom-right alignment: key j visible to row i iff
    j <= i + N_k - N_q): PyTorch SDPA (CPU, float64) with that explicit mask
    on every row that sees a key; rows that see none (N_q > N_k) give O = 0 and
    LSE = -inf; with N_q == N_k it is the top-left mask."""
    for (Nq, Nk, seed) in [(9, 21, 60), (21, 9, 61), (13, 13, 62)]:
        Q, K, V = _rand((Nq, 8), seed), _rand((Nk, 8), seed + 1), _rand((Nk, 8), seed + 2)
        O, L = attn(Q, K, V, 0.3, 2)
        mask = torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
        tq, tk, tv = (torch.from_numpy(x.astype(np.float64)) for x in (Q, K, V))
        seen = mask.any(1).numpy()
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq[None, seen], tk[None], tv[None], attn_mask=mask[seen], scale=0.3)[0]
        S = (0.3 * tq @ tk.T).masked_fill(~mask, float("-inf"))
        np.testing.assert_allclose(O[seen], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[seen], torch.logsumexp(S[seen], -1).numpy(), rtol=0, atol=1e-12)
        assert np.all(O[~seen] == 0.0) and np.all(np.isneginf(L[~seen]))
        if Nq == Nk:
            O1, L1 = attn(Q, K, V, 0.3, True)
            np.testing.assert_allclose(O, O1, rtol=0, atol=1e-12)


PINS = [pin_q_zero, pin_scale_zero, pin_single_key, pin_first_causal_row,
        pin_permutation, pin_large_scores, pin_online_softmax_recompute,
        pin_torch_sdpa, pin_invariants, pin_worked_examples, pin_bottom_right_causal]


# ----------------------------------------------------------------------------
# the oracle against every pin
# ----------------------------------------------------------------------------

@pytest.fixture(scope="module")
def oracle_attn(oracle_mod):
    def attn(Q, K, V, scale, causal):
        return oracle_mod.attention(Q, K, V, scale, causal)
    return attn


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle_attn):
    pin(oracle_attn)


def test_oracle_batched_and_row_subset(oracle_mod):
    """Leading [B, H] dims loop over slices; a row subset equals those rows
    of the full evaluation."""
    Q, K, V = _rand((2, 3, 10, 4), 50), _rand((2, 3, 12, 4), 51), _rand((2, 3, 12, 4), 52)
    O, L = oracle_mod.attention(Q, K, V, 0.5, True)
    assert O.shape == (2, 3, 10, 4) and L.shape == (2, 3, 10)
    O1, L1 = oracle_mod.attention(Q[1, 2], K[1, 2], V[1, 2], 0.5, True)
    np.testing.assert_array_equal(O[1, 2], O1)
    rows = [9, 0, 4]
    Os, Ls = oracle_mod.attention(Q, K, V, 0.5, True, rows=rows)
    np.testing.assert_array_equal(Os, O[..., rows, :])
    np.testing.assert_array_equal(Ls, L[..., rows])


def test_oracle_regression_fixture(oracle_mod):
    """The stored seeded fixture (written by tests/golden/make_golden.py, which
    calls only the oracle) still matches: guards against silent edits."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", GOLDEN / "make_golden.py")
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    data = json.loads((GOLDEN / "oracle_seeded.json").read_text())
    for case in data["cases"]:
        Q, K, V = mg.case_inputs(case)
        O, L = oracle_mod.attention(Q, K, V, case["scale"], case["causal"])
        np.testing.assert_allclose(O.reshape(-1)[:64], case["O_head"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(L.reshape(-1)[:64], case["LSE_head"], rtol=0, atol=1e-13)
        assert abs(float(O.sum()) - case["O_sum"]) <= 1e-9
        assert abs(float(L.sum()) - case["LSE_sum"]) <= 1e-9


# ----------------------------------------------------------------------------
# the pins are strong enough: each plausible mistake trips at least one
# ----------------------------------------------------------------------------

def _mutant(kind):
    def attn(Q, K, V, scale, causal):
        Q = Q.astype(np.float64)
        K = K.astype(np.float64)
        V = V.astype(np.float64)
        Nq, Nk = Q.shape[0], K.shape[0]
        sc = 1.0 if kind == "no_scale" else scale
        S = sc * (Q @ K.T)
        if kind == "transposed_scores" and Nq == Nk:
            S = S.T
        if kind == "negated_scores":
            S = -S
        i = np.arange(Nq)[:, None]
        j = np.arange(Nk)[None, :]
        if causal is not True and causal == 2:  # bottom-right alignment
            off = Nk - Nq
            if kind == "bottom_right_sign":
                off = Nq - Nk
            vis = j <= i + off
            S = np.where(vis, S, -np.inf)
        elif causal:
            if kind == "causal_strict":
                vis = j < i
            elif kind == "causal_bottom_right":
                vis = j <= i + (Nk - Nq)
            else:
                vis = j <= i
            S = np.where(vis, S, -np.inf)
        empty = np.all(np.isneginf(S), axis=1)  # rows that see no key: O = 0, LSE = -inf
        S = np.where(empty[:, None], 0.0, S)
        if kind == "no_max_shift":
            with np.errstate(over="ignore", invalid="ignore"):
                P = np.exp(S)
                l = P.sum(1)
                return (P @ V) / l[:, None], np.log(l)
        m = S.max(1)
        P = np.exp(S - m[:, None])
        l = P.sum(1)
        O = (P @ V) if kind == "no_normalise" else (P @ V) / l[:, None]
        L = m + (np.log2(l) if kind == "lse_log2" else np.log(l))
        if kind == "lse_missing_max":
            L = np.log(l)
        if kind == "v_is_k":
            O = (P @ K) / l[:, None]
        if kind != "bottom_right_empty_rows_mean":
            O = np.where(empty[:, None], 0.0, O)
            L = np.where(empty, -np.inf, L)
        return O, L
    return attn


MUTANTS = ["no_scale", "transposed_scores", "negated_scores", "causal_strict",
           "causal_bottom_right", "no_max_shift", "no_normalise", "lse_log2",
           "lse_missing_max", "v_is_k", "bottom_right_sign", "bottom_right_empty_rows_mean"]


def test_correct_reference_passes_all_pins():
    """The mutant harness itself, with no mutation, passes every pin."""
    for pin in PINS:
        pin(_mutant("none"))


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_mistake_trips_a_pin(kind):
    attn = _mutant(kind)
    tripped = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(attn)
        except (AssertionError, FloatingPointError, ValueError):
            tripped.append(pin.__name__)
    assert tripped, f"mutant {kind} passed every pin"
