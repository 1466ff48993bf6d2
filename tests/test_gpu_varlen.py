"""Packed variable-length batches through fa_fwd_varlen, against the oracle's
packed attention (each sequence its own problem, the causal alignment per
sequence), element by element.

The lengths cover an empty sequence, single rows, the 256-row query tile and
the 128-key tile on both sides of their edges, lengths spanning several tiles
with a ragged tail, key ranges shorter and longer than the query range
(cross attention, bottom-right rows that see no key), grouped K/V heads, the
packed QKV layout (q, k, v as strided slices of one [total, 3, H, d] tensor)
and a loose max_seqlen_q bound.  Every packed row of O and LSE is written:
the outputs start as NaN."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, packed, seq_lengths

pytestmark = pytest.mark.gpu
TOL_O, TOL_LSE = 2e-2, 1e-2  # bf16 inputs and output, fp32 accumulation


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _check(oracle_mod, q, k, v, cu_q, cu_k, causal, d, max_len=None, H_kv=None, layout=None):
    H = q.shape[1]
    G = H // k.shape[1]
    scale = 1.0 / math.sqrt(d)
    lens_q = (cu_q[1:] - cu_q[:-1]).tolist()
    max_len = max_len or max(max(lens_q), 1)
    if layout is not None:
        qd, kd, vd = layout
    else:
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    O = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    L = torch.full((H, q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    fa.fwd_varlen(qd, kd, vd, cu_q.cuda(), cu_k.cuda(), max_len, scale=scale, is_causal=causal, out=O, lse=L)
    fa.check()
    kx = k.float().repeat_interleave(G, dim=1).numpy()
    vx = v.float().repeat_interleave(G, dim=1).numpy()
    O_ref, L_ref = oracle_mod.attention_varlen(q.float().numpy(), kx, vx, cu_q.numpy(), cu_k.numpy(), scale,
                                               fa.causal_code(causal))
    Og, Lg = O.float().cpu().numpy(), L.cpu().numpy()
    assert np.isfinite(Og).all(), "a packed output row was not written"
    assert not np.isnan(Lg).any(), "a packed LSE entry was not written"
    assert np.array_equal(np.isneginf(Lg), np.isneginf(L_ref)), "rows without keys differ"
    fin = np.isfinite(L_ref)
    eo = float(np.abs(Og - O_ref).max(initial=0.0))
    el = float(np.abs(Lg[fin] - L_ref[fin]).max(initial=0.0))
    assert eo <= TOL_O and el <= TOL_LSE, f"max|dO|={eo:.3e} max|dLSE|={el:.3e}"


LENGTHS = {
    "edges": ([0, 1, 255, 256, 257, 129, 513], [0, 1, 255, 256, 257, 129, 513]),
    "cross": ([300, 17, 1000, 64], [128, 700, 333, 1]),
    "no_keys": ([40, 300, 2], [0, 90, 7]),
    "long_tail": ([1000, 3, 611], [1000, 3, 611]),
}


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"], ids=["nc", "top_left", "bottom_right"])
@pytest.mark.parametrize("case", list(LENGTHS))
def test_varlen_forward(oracle_mod, d, causal, case):
    lq, lk = LENGTHS[case]
    q, k, v, cu_q, cu_k = packed(lq, lk, 3, 3, d, 1300 + d + len(case), torch.bfloat16)
    _check(oracle_mod, q, k, v, cu_q, cu_k, causal, d)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(6, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"], ids=["nc", "top_left", "bottom_right"])
def test_varlen_gqa(oracle_mod, d, H, H_kv, causal):
    lq, lk = [200, 513, 0, 77], [260, 300, 5, 77]
    q, k, v, cu_q, cu_k = packed(lq, lk, H, H_kv, d, 1400 + d + H_kv, torch.bfloat16)
    _check(oracle_mod, q, k, v, cu_q, cu_k, causal, d)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_varlen_packed_qkv_layout_and_loose_bound(oracle_mod, causal):
    # q, k, v as slices of one packed [total, 3, H, d] tensor; max_seqlen_q well above the true maximum
    lens = [333, 128, 900, 1]
    H, d = 4, 128
    total = sum(lens)
    qkv = normal((total, 3, H, d), 1500, torch.bfloat16)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    dev = qkv.cuda()
    _check(oracle_mod, qkv[:, 0], qkv[:, 1], qkv[:, 2], cu, cu, causal, d, max_len=1300,
           layout=(dev[:, 0], dev[:, 1], dev[:, 2]))


def test_varlen_equal_lengths_match_batched():
    # equal lengths: the packed call and the batched [B, H, N, d] call compute the same rows
    B, H, N, d = 3, 4, 700, 128
    q, k, v, cu_q, cu_k = packed([N] * B, [N] * B, H, H, d, 1600, torch.bfloat16)
    for causal in (False, True):
        O, L = fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), N, is_causal=causal)
        qb = q.cuda().reshape(B, N, H, d).transpose(1, 2)
        kb = k.cuda().reshape(B, N, H, d).transpose(1, 2)
        vb = v.cuda().reshape(B, N, H, d).transpose(1, 2)
        Ob, Lb = fa.fwd(qb, kb, vb, is_causal=causal, split_kv=1)
        fa.check()
        assert torch.equal(O, Ob.transpose(1, 2).reshape(B * N, H, d))
        assert torch.equal(L, Lb.permute(1, 0, 2).reshape(H, B * N))


def test_varlen_many_sequences_sampled(oracle_mod):
    # a mixed-length batch of the benchmark's shape (H = 32, d = 128): sampled sequences checked
    lens = seq_lengths(24, 64, 4096, 1700)
    H, d = 32, 128
    q, k, v, cu_q, cu_k = packed(lens, lens, H, H, d, 1700, torch.bfloat16)
    O, L = fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), max(lens), is_causal=True)
    fa.check()
    Og, Lg = O.float().cpu().numpy(), L.cpu().numpy()
    assert np.isfinite(Og).all() and np.isfinite(Lg).all()
    scale = 1.0 / math.sqrt(d)
    for b in (0, 7, 23):
        s0, s1 = int(cu_q[b]), int(cu_q[b + 1])
        rows = np.unique(np.r_[0, s1 - s0 - 1, np.linspace(0, s1 - s0 - 1, 9).astype(int)])
        for h in (0, 31):
            Or, Lr = oracle_mod.attention(q[s0:s1, h].float().numpy(), k[s0:s1, h].float().numpy(),
                                          v[s0:s1, h].float().numpy(), scale, True, rows=rows)
            assert float(np.abs(Og[s0 + rows, h] - Or).max()) <= TOL_O
            assert float(np.abs(Lg[h, s0 + rows] - Lr).max()) <= TOL_LSE


def test_varlen_rejects_bad_arguments():
    q, k, v, cu_q, cu_k = packed([10, 20], [10, 20], 2, 2, 128, 1800, torch.bfloat16)
    qd, kd, vd, cq, ck = q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda()
    with pytest.raises(ValueError):
        fa.fwd_varlen(qd, kd, vd, cq.long(), ck, 20)          # offsets must be int32
    with pytest.raises(ValueError):
        fa.fwd_varlen(qd, kd, vd, cq[:2], ck, 20)             # B + 1 offsets on both sides
    with pytest.raises(fa.FaError):
        fa.fwd_varlen(qd, kd, vd, cq, ck, 31)                 # max_seqlen_q above total_q
    with pytest.raises(fa.FaError):
        fa.fwd_varlen(qd.float(), kd.float(), vd.float(), cq, ck, 20)  # bf16 only


def test_varlen_concurrent_streams_and_back_to_back(oracle_mod):
    """Packed batches take their work units from per-launch counters (one of
    64 slots, round robin, zeroed by each launch's last CTA): launches in
    flight at once on four streams, and many back to back on one stream, must
    each cover every unit exactly once -- every output equals the one-launch
    result bit for bit, and that one matches the oracle."""
    cases = []
    for i, (lens, causal) in enumerate((([300, 700, 129, 1000], False), ([513, 64, 900], True),
                                        ([1, 256, 257, 640], "bottom_right"), ([1200, 90], False))):
        q, k, v, cu_q, cu_k = packed(lens, lens, 4, 2, 128, seed=7100 + i)
        cases.append((q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), max(lens), causal))
    refs = []
    for q, k, v, cq, ck, ml, causal in cases:
        O, L = fa.fwd_varlen(q, k, v, cq, ck, ml, is_causal=causal)
        fa.check()
        refs.append((O.clone(), L.clone()))
    # the first case against the oracle as well
    q, k, v, cq, ck, ml, causal = cases[0]
    kx = k.float().repeat_interleave(2, dim=1).cpu().numpy()
    vx = v.float().repeat_interleave(2, dim=1).cpu().numpy()
    O_ref, L_ref = oracle_mod.attention_varlen(q.float().cpu().numpy(), kx, vx, cq.cpu().numpy(), ck.cpu().numpy(),
                                               1 / math.sqrt(128), fa.causal_code(causal))
    assert float(np.abs(refs[0][0].float().cpu().numpy() - O_ref).max()) <= TOL_O
    # four streams at once, several rounds
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [[None] * len(cases) for _ in range(3)]
    torch.cuda.synchronize()
    for r in range(3):
        for c, (q, k, v, cq, ck, ml, causal) in enumerate(cases):
            with torch.cuda.stream(streams[c]):
                outs[r][c] = fa.fwd_varlen(q, k, v, cq, ck, ml, is_causal=causal, stream=streams[c])
    torch.cuda.synchronize()
    fa.check()
    for r in range(3):
        for c in range(len(cases)):
            assert torch.equal(outs[r][c][0], refs[c][0]) and torch.equal(outs[r][c][1], refs[c][1]), (r, c)
    # 100 launches back to back on one stream (every slot taken and reset more than once)
    q, k, v, cq, ck, ml, causal = cases[1]
    for _ in range(100):
        O, L = fa.fwd_varlen(q, k, v, cq, ck, ml, is_causal=causal)
    fa.check()
    assert torch.equal(O, refs[1][0]) and torch.equal(L, refs[1][1])

@pytest.mark.parametrize("causal", [False, True], ids=["nc", "top_left"])
def test_varlen_output_view_inside_wider_buffer(oracle_mod, causal):
    """Packed O as a view into a larger buffer (row pitch H x (d + 24), spare
    rows after the last sequence).  Sequence ends fall inside 32-row blocks,
    so some warps store by TMA and the one straddling each end row by row:
    every packed row of the view is written and nothing outside it."""
    d, H = 128, 3
    lq = [300, 17, 129, 64]
    q, k, v, cu_q, cu_k = packed(lq, lq, H, H, d, 1777, torch.bfloat16)
    total = q.shape[0]
    big = torch.full((total + 7, H, d + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    O = big[:total, :, :d]
    O.fill_(float("nan"))
    L = torch.full((H, total), float("nan"), dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), max(lq), scale=scale,
                  is_causal=causal, out=O, lse=L)
    fa.check()
    O_ref, L_ref = oracle_mod.attention_varlen(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                               cu_q.numpy(), cu_k.numpy(), scale, fa.causal_code(causal))
    Og = O.float().cpu().numpy()
    assert np.isfinite(Og).all(), "a packed output row was not written"
    eo = float(np.abs(Og - O_ref).max())
    el = float(np.abs(L.cpu().numpy() - L_ref).max())
    assert eo <= TOL_O and el <= TOL_LSE, f"max|dO|={eo:.3e} max|dLSE|={el:.3e}"
    assert bool((big[total:] == 7).all()), "a store wrote past the last packed row"
    assert bool((big[:total, :, d:] == 7).all()), "a store wrote past the view's last column"
