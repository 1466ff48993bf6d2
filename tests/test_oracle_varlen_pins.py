"""Pins of the oracle's packed variable-length attention (``oracle.attention_varlen``).

A packed batch is B sequences of different lengths laid end to end, sequence b
at rows cu[b] .. cu[b+1]-1; each attends to its own keys only, with the causal
alignment (top-left or bottom-right) taken per sequence.  The pins check the
oracle against things fixed independently of its slicing code:

* equal lengths reduce to the batched definition [B, H, N, d] (itself pinned
  against closed forms and brute force);
* a single sequence is plain attention;
* brute force over the whole packed batch with a block-diagonal mask (a
  dense softmax over all packed keys, masked to the query's own sequence);
* permuting the sequences permutes the outputs;
* a sequence's outputs do not depend on another sequence's keys;
* rows that see no key (an empty key range, or bottom-right alignment with
  more queries than keys) give O = 0 and LSE = -inf.

Each plausible slicing mistake (global causal indices, one key too many, no
block-diagonal mask, bottom-right offset from the packed totals, NaN rows)
trips at least one pin (mutants at the end).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

rng = np.random.default_rng(20261202)


def _pack(lens_q, lens_k, H, d, seed):
    g = np.random.default_rng(seed)
    cq = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    q = g.standard_normal((int(cq[-1]), H, d)).astype(np.float32)
    k = g.standard_normal((int(ck[-1]), H, d)).astype(np.float32)
    v = g.standard_normal((int(ck[-1]), H, d)).astype(np.float32)
    return q, k, v, cq, ck


def _brute(q, k, v, cq, ck, scale, causal, kind="none"):
    """Dense softmax over every packed key, masked to the query's own sequence."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    Tq, H, d = q.shape
    Tk = k.shape[0]
    sq = np.searchsorted(cq, np.arange(Tq), side="right") - 1  # sequence of each packed row
    sk = np.searchsorted(ck, np.arange(Tk), side="right") - 1
    iq = np.arange(Tq) - cq[sq]                                 # index inside its sequence
    jk = np.arange(Tk) - ck[sk]
    if kind == "global_causal":
        iq, jk = np.arange(Tq), np.arange(Tk)
    same = sq[:, None] == sk[None, :]
    if kind == "shared_keys":
        same = np.ones_like(same)
    if kind == "one_more_key":  # the key just past the sequence's end is visible too
        same = same | ((sk[None, :] == sq[:, None] + 1) & (jk[None, :] == 0))
    vis = same
    if causal:
        off = np.zeros(Tq, dtype=np.int64)
        if causal == 2:
            lq = (cq[1:] - cq[:-1])[sq]
            lk = (ck[1:] - ck[:-1])[sq]
            off = lk - lq
            if kind == "bottom_right_totals":
                off = np.full(Tq, Tk - Tq)
        vis = vis & (jk[None, :] <= iq[:, None] + off[:, None])
    O = np.zeros((Tq, H, d))
    L = np.full((H, Tq), -np.inf)
    for h in range(H):
        S = scale * q[:, h] @ k[:, h].T
        S = np.where(vis, S, -np.inf)
        empty = ~vis.any(1)
        S = np.where(empty[:, None], 0.0, S)
        m = S.max(1)
        P = np.exp(S - m[:, None]) * vis
        l = P.sum(1)
        with np.errstate(invalid="ignore", divide="ignore"):
            Oh = (P @ v[:, h]) / l[:, None]
            Lh = m + np.log(l)
        if kind != "nan_empty_rows":
            Oh = np.where(empty[:, None], 0.0, Oh)
            Lh = np.where(empty, -np.inf, Lh)
        O[:, h] = Oh
        L[h] = Lh
    return O, L


def _close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin) and np.array_equal(a[~fin], b[~fin])
    assert float(np.abs(a[fin] - b[fin]).max(initial=0.0)) <= tol


CASES = [  # (lens_q, lens_k): ragged, empty sequences, no keys, more queries than keys
    ([5, 0, 9, 1, 7], [5, 3, 9, 1, 7]),
    ([4, 6, 3], [7, 2, 0]),
    ([8, 2], [3, 11]),
]


def pin_equal_lengths_match_batched(f):
    B, H, N, d = 3, 2, 11, 8
    q, k, v, cq, ck = _pack([N] * B, [N] * B, H, d, 11)
    for causal in (0, 1, 2):
        O, L = f(q, k, v, cq, ck, 0.3, causal)
        Ob, Lb = oracle.attention(q.reshape(B, N, H, d).transpose(0, 2, 1, 3),
                                  k.reshape(B, N, H, d).transpose(0, 2, 1, 3),
                                  v.reshape(B, N, H, d).transpose(0, 2, 1, 3), 0.3, causal)
        _close(O, Ob.transpose(0, 2, 1, 3).reshape(B * N, H, d))
        _close(L, Lb.transpose(1, 0, 2).reshape(H, B * N))


def pin_single_sequence_is_attention(f):
    q, k, v, cq, ck = _pack([13], [9], 2, 8, 12)
    for causal in (0, 1, 2):
        O, L = f(q, k, v, cq, ck, 0.5, causal)
        Ob, Lb = oracle.attention(q.transpose(1, 0, 2), k.transpose(1, 0, 2), v.transpose(1, 0, 2), 0.5, causal)
        _close(O, Ob.transpose(1, 0, 2))
        _close(L, Lb)


def pin_block_diagonal_brute_force(f):
    for n, (lq, lk) in enumerate(CASES):
        q, k, v, cq, ck = _pack(lq, lk, 2, 8, 20 + n)
        for causal in (0, 1, 2):
            O, L = f(q, k, v, cq, ck, 0.35, causal)
            Ob, Lb = _brute(q, k, v, cq, ck, 0.35, causal)
            _close(O, Ob, 1e-11)
            _close(L, Lb, 1e-11)


def pin_sequence_permutation(f):
    lq, lk = [5, 8, 3, 6], [7, 8, 2, 9]
    q, k, v, cq, ck = _pack(lq, lk, 2, 8, 30)
    perm = [2, 0, 3, 1]

    def reorder(x, cu, lens):
        return np.concatenate([x[cu[b]:cu[b + 1]] for b in perm]), \
            np.concatenate([[0], np.cumsum([lens[b] for b in perm])]).astype(np.int32)
    for causal in (0, 1, 2):
        O, L = f(q, k, v, cq, ck, 0.4, causal)
        q2, cq2 = reorder(q, cq, lq)
        k2, ck2 = reorder(k, ck, lk)
        v2, _ = reorder(v, ck, lk)
        O2, L2 = f(q2, k2, v2, cq2, ck2, 0.4, causal)
        Or, _ = reorder(O, cq, lq)
        Lr = np.concatenate([L[:, cq[b]:cq[b + 1]] for b in perm], axis=1)
        _close(O2, Or)
        _close(L2, Lr)


def pin_other_sequences_do_not_matter(f):
    lq, lk = [6, 5, 7], [6, 4, 9]
    q, k, v, cq, ck = _pack(lq, lk, 2, 8, 40)
    for causal in (0, 1, 2):
        O, L = f(q, k, v, cq, ck, 0.4, causal)
        k2, v2 = k.copy(), v.copy()
        k2[ck[1]:] = rng.standard_normal(k2[ck[1]:].shape)  # keys of sequences 1 and 2 change
        v2[ck[1]:] = rng.standard_normal(v2[ck[1]:].shape)
        O2, L2 = f(q, k2, v2, cq, ck, 0.4, causal)
        _close(O2[:cq[1]], O[:cq[1]])
        _close(L2[:, :cq[1]], L[:, :cq[1]])
        assert not np.allclose(O2[cq[1]:], O[cq[1]:])


def pin_rows_without_keys(f):
    q, k, v, cq, ck = _pack([3, 6], [0, 2], 1, 4, 50)
    O, L = f(q, k, v, cq, ck, 1.0, 0)
    assert np.all(O[:3] == 0) and np.all(np.isneginf(L[:, :3]))   # sequence 0 has no keys
    O, L = f(q, k, v, cq, ck, 1.0, 2)  # bottom-right: row i of sequence 1 sees keys j <= i - 4
    assert np.all(O[3:7] == 0) and np.all(np.isneginf(L[:, 3:7]))
    assert np.all(np.isfinite(L[:, 7:]))
    np.testing.assert_allclose(O[7, 0], v[0, 0], rtol=0, atol=1e-12)  # the first visible row sees key 0 alone
    np.testing.assert_allclose(L[0, 7], float(q[7, 0].astype(np.float64) @ k[0, 0].astype(np.float64)),
                               rtol=0, atol=1e-12)


PINS = [pin_equal_lengths_match_batched, pin_single_sequence_is_attention, pin_block_diagonal_brute_force,
        pin_sequence_permutation, pin_other_sequences_do_not_matter, pin_rows_without_keys]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_varlen_oracle_pin(pin):
    pin(oracle.attention_varlen)


def test_varlen_oracle_rejects_bad_offsets():
    q, k, v, cq, ck = _pack([3, 4], [3, 4], 1, 4, 60)
    with pytest.raises(ValueError):
        oracle.attention_varlen(q, k, v, np.array([0, 4, 3], np.int32), ck, 1.0)
    with pytest.raises(ValueError):
        oracle.attention_varlen(q, k, v, cq, np.array([0, 3, 8], np.int32), 1.0)


MUTANTS = ["global_causal", "shared_keys", "one_more_key", "bottom_right_totals", "nan_empty_rows"]


def test_brute_force_harness_passes_all_pins():
    for pin in PINS:
        pin(lambda *a: _brute(*a))


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_varlen_mistake_trips_a_pin(kind):
    def f(q, k, v, cq, ck, scale, causal):
        return _brute(q, k, v, cq, ck, scale, causal, kind)
    tripped = []
    for pin in PINS:
        if pin is pin_block_diagonal_brute_force:
            continue  # it compares against the unmutated harness: count only the independent pins
        try:
            with np.errstate(all="ignore"):
                pin(f)
        except (AssertionError, FloatingPointError, ValueError):
            tripped.append(pin.__name__)
    assert tripped, f"mutant {kind} passed every independent pin"
