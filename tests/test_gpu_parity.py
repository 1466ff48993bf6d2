"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs.

Tolerances (max-abs error):
  bf16 inputs (tcgen05 kind::f16):      O <= 2e-2, LSE <= 1e-2
  fp32 inputs (tcgen05 kind::tf32, and the fp32 small-head path):
                                        O <= 3e-3, LSE <= 2e-3
Outputs are pre-filled with NaN so that an element the kernel never writes
fails the comparison.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import AXIAL, WORKLOADS, normal, qkv

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float32: (3e-3, 2e-3)}


@pytest.fixture(scope="module", autouse=True)
def _setup(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _poisoned(shape, dtype):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def run_gpu(Q, K, V, scale, causal, split_kv=None):
    """Q, K, V on the host -> (O, LSE) from the GPU, as host tensors.
    split_kv=None lets the library choose (long key ranges over few query
    tiles are then split)."""
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    O = _poisoned(Q.shape, Q.dtype)
    L = _poisoned(Q.shape[:-1], torch.float32)
    fa.fwd(Qd, Kd, Vd, scale=scale, is_causal=causal, out=O, lse=L, split_kv=split_kv)
    fa.check()
    return O.float().cpu().numpy(), L.cpu().numpy()


def assert_close(O, L, O_ref, L_ref, dtype, what=""):
    to, tl = TOL[dtype]
    assert np.isfinite(O).all() and np.isfinite(L).all(), f"{what}: non-finite output"
    eo = float(np.abs(O - O_ref).max())
    el = float(np.abs(L - L_ref).max())
    assert eo <= to and el <= tl, f"{what}: max|dO|={eo:.3e} (tol {to}) max|dLSE|={el:.3e} (tol {tl})"
    return eo, el


# ---------------------------------------------------------------- ragged shapes
SHAPES = [(1, 1), (17, 17), (100, 100), (129, 129), (255, 255), (256, 256), (257, 257),
          (300, 300), (513, 513), (100, 300), (300, 100), (257, 1000), (64, 777)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("nq,nk", SHAPES)
def test_tensor_core_ragged(oracle_mod, dtype, d, causal, nq, nk):
    seed = 1000 + nq * 7 + nk * 13 + d + (1 if causal else 0)
    Q, K, V = qkv((2, 3, nq, d), (2, 3, nk, d), seed, dtype)
    scale = 1.0 / math.sqrt(d)
    O, L = run_gpu(Q, K, V, scale, causal, split_kv=1)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, causal)
    assert_close(O, L, O_ref, L_ref, dtype, f"{dtype} d={d} {nq}x{nk} causal={causal}")


# ------------------------------------------------------------------ split-KV
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("nq,nk,split", [(300, 1000, 1), (300, 1000, 2), (257, 1000, 3), (100, 777, 5),
                                         (513, 513, 2), (64, 129, 2), (1, 300, 3)])
def test_split_kv_ragged(oracle_mod, dtype, d, causal, nq, nk, split):
    """Forced split counts (1 = the plain path), ragged lengths, causal rows
    whose keys fall outside some splits."""
    Q, K, V = qkv((2, 2, nq, d), (2, 2, nk, d), 3000 + nq + nk + split + d, dtype)
    scale = 1.0 / math.sqrt(d)
    O, L = run_gpu(Q, K, V, scale, causal, split_kv=split)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, causal)
    assert_close(O, L, O_ref, L_ref, dtype, f"split={split} {dtype} d={d} {nq}x{nk} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq,nk", [(300, 4096), (256, 5000)])
def test_auto_split_long_keys(oracle_mod, d, nq, nk):
    """A few query tiles over a long key range: the library's own choice
    splits the keys (bf16, non-causal), and the merged result matches."""
    B, H = 1, 2
    n = fa.lib().fa_fwd_splitkv_choose(fa.FA_BF16, B, H, nq, nk, d, 0)
    assert n > 1
    assert fa.lib().fa_fwd_splitkv_choose(fa.FA_BF16, B, H, nq, nk, d, 1) == 1   # causal: never
    assert fa.lib().fa_fwd_splitkv_choose(fa.FA_FP32, B, H, nq, nk, d, 0) == 1   # tf32: never
    Q, K, V = qkv((B, H, nq, d), (B, H, nk, d), 4000 + nq + nk + d, torch.bfloat16)
    O, L = run_gpu(Q, K, V, 1.0 / math.sqrt(d), False, split_kv=None)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, 1.0 / math.sqrt(d), False)
    assert_close(O, L, O_ref, L_ref, torch.bfloat16, f"auto split={n} d={d} {nq}x{nk}")


def test_split_kv_strided_and_workspace_reuse(oracle_mod):
    """Head-major strided storage through the split path, two calls sharing
    one caller-provided workspace."""
    B, H, N, Nk, d = 2, 4, 200, 900, 128
    Qs, Ks, Vs = normal((B, N, H, d), 61, torch.bfloat16), normal((B, Nk, H, d), 62, torch.bfloat16), \
        normal((B, Nk, H, d), 63, torch.bfloat16)
    need = fa.lib().fa_fwd_splitkv_workspace_bytes(B, H, N, d, 3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for causal in (False, True):
        Od = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
        Ld = _poisoned((B, H, N), torch.float32)
        fa.fwd(Qs.cuda().transpose(1, 2), Ks.cuda().transpose(1, 2), Vs.cuda().transpose(1, 2),
               scale=0.09, is_causal=causal, out=Od, lse=Ld, split_kv=3, workspace=ws)
        fa.check()
        O_ref, L_ref = oracle_mod.attention(Qs.transpose(1, 2), Ks.transpose(1, 2), Vs.transpose(1, 2),
                                            0.09, causal)
        assert_close(Od.float().cpu().numpy(), Ld.cpu().numpy(), O_ref, L_ref, torch.bfloat16,
                     f"split strided causal={causal}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("d", [16, 32])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("nq,nk", [(1, 1), (32, 32), (31, 45), (100, 70), (64, 200)])
def test_small_head_ragged(oracle_mod, dtype, d, causal, nq, nk):
    Q, K, V = qkv((2, 3, nq, d), (2, 3, nk, d), 2000 + nq + nk + d, dtype)
    scale = 1.0 / math.sqrt(d)
    O, L = run_gpu(Q, K, V, scale, causal)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, causal)
    assert_close(O, L, O_ref, L_ref, torch.float32 if dtype == torch.float32 else dtype,
                 f"small {dtype} d={d} {nq}x{nk} causal={causal}")


@pytest.mark.parametrize("d,causal", [(128, False), (128, True), (64, False)], ids=["d128_nc", "d128_causal", "d64_nc"])
def test_output_view_inside_wider_buffer(oracle_mod, d, causal):
    """O as a view into a larger buffer (row pitch d + 24, five spare rows per
    head) with a ragged N: the tiles' O stores (TMA stores clipped to the
    view) write every element of the view and nothing outside it."""
    B, H, N = 2, 3, 300
    Q = normal((B, H, N, d), 41, torch.bfloat16)
    K = normal((B, H, N, d), 42, torch.bfloat16)
    V = normal((B, H, N, d), 43, torch.bfloat16)
    big = torch.full((B, H, N + 5, d + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    O = big[:, :, :N, :d]
    O.fill_(float("nan"))
    L = _poisoned((B, H, N), torch.float32)
    fa.fwd(Q.cuda(), K.cuda(), V.cuda(), scale=0.1, is_causal=causal, out=O, lse=L)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q, K, V, 0.1, causal)
    assert_close(O.float().cpu().numpy(), L.cpu().numpy(), O_ref, L_ref, torch.bfloat16, f"view d={d}")
    assert bool((big[:, :, N:, :] == 7).all()), "a store wrote past the view's last row"
    assert bool((big[:, :, :N, d:] == 7).all()), "a store wrote past the view's last column"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_strided_heads_major_layout(oracle_mod, dtype):
    """Q, K, V, O as [B, N, H, d] storage viewed as [B, H, N, d] (non-monotonic strides)."""
    B, H, N, d = 2, 4, 333, 128
    Qs = normal((B, N, H, d), 31, dtype)
    Ks = normal((B, N, H, d), 32, dtype)
    Vs = normal((B, N, H, d), 33, dtype)
    Q, K, V = (x.transpose(1, 2) for x in (Qs, Ks, Vs))
    Od = torch.full((B, N, H, d), float("nan"), dtype=dtype, device="cuda").transpose(1, 2)
    Ld = _poisoned((B, H, N), torch.float32)
    fa.fwd(Qs.cuda().transpose(1, 2), Ks.cuda().transpose(1, 2), Vs.cuda().transpose(1, 2),
           scale=0.09, is_causal=True, out=Od, lse=Ld)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q.contiguous(), K.contiguous(), V.contiguous(), 0.09, True)
    assert_close(Od.float().cpu().numpy(), Ld.cpu().numpy(), O_ref, L_ref, dtype, "strided")


@pytest.mark.parametrize("scale", [0.0, -0.2, 2.0])
def test_unusual_scales(oracle_mod, scale):
    Q, K, V = qkv((1, 2, 200, 64), (1, 2, 333, 64), 41, torch.bfloat16)
    O, L = run_gpu(Q, K, V, scale, False)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, False)
    assert_close(O, L, O_ref, L_ref, torch.bfloat16, f"scale={scale}")


def test_q_zero_closed_form():
    """Q = 0 on the GPU: O = mean of V rows, LSE = log N_k (causal: prefix means)."""
    N = 300
    Q = torch.zeros(1, 1, N, 128, dtype=torch.bfloat16)
    V = normal((1, 1, N, 128), 51, torch.bfloat16)
    K = normal((1, 1, N, 128), 52, torch.bfloat16)
    O, L = run_gpu(Q, K, V, 0.1, True)
    Vd = V.double().numpy()[0, 0]
    pref = np.cumsum(Vd, axis=0) / np.arange(1, N + 1)[:, None]
    assert np.abs(O[0, 0] - pref).max() <= 2e-2
    assert np.abs(L[0, 0] - np.log(np.arange(1, N + 1))).max() <= 1e-2
    assert np.abs(O[0, 0, 0] - Vd[0]).max() <= 8e-3  # first causal row is V[0]


def test_lse_optional_and_no_lse_write():
    Q, K, V = (x.cuda() for x in qkv((1, 2, 130, 64), (1, 2, 130, 64), 61, torch.bfloat16))
    O1, L1 = fa.fwd(Q, K, V, with_lse=False)
    O2, L2 = fa.fwd(Q, K, V)
    fa.check()
    assert L1 is None and L2 is not None
    assert torch.equal(O1, O2)


def test_deterministic():
    Q, K, V = (x.cuda() for x in qkv((2, 4, 700, 128), (2, 4, 700, 128), 71, torch.bfloat16))
    O1, L1 = fa.fwd(Q, K, V, is_causal=True)
    O2, L2 = fa.fwd(Q, K, V, is_causal=True)
    fa.check()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


# -------------------------------------------------------- the five configurations
def _cfg_full(oracle_mod, name):
    w = WORKLOADS[name]
    Q, K, V = w.make()
    O, L = run_gpu(Q, K, V, w.scale, w.causal)
    O_ref, L_ref = oracle_mod.attention(Q, K, V, w.scale, w.causal)
    return assert_close(O, L, O_ref, L_ref, w.dtype, name)


@pytest.mark.parametrize("name", ["tiny_nc", "tiny_causal", "tutorial_nc", "tutorial_causal"])
def test_config_full(oracle_mod, name):
    _cfg_full(oracle_mod, name)


def test_config_axial(oracle_mod):
    w = AXIAL
    Q, K, V = w.make()
    (O_row, L_row), (O_col, L_col) = fa.axial(Q.cuda(), K.cuda(), V.cuda(), scale=w.scale, with_lse=True)
    fa.check()
    # row attention: sequences along Wg for each (b, hg, head)
    qr = Q.permute(0, 1, 3, 2, 4)
    O_ref, L_ref = oracle_mod.attention(qr, K.permute(0, 1, 3, 2, 4), V.permute(0, 1, 3, 2, 4), w.scale)
    assert_close(O_row.permute(0, 1, 3, 2, 4).cpu().numpy(), L_row.permute(0, 1, 3, 2).cpu().numpy(),
                 O_ref, L_ref, torch.float32, "axial row")
    # column attention: sequences along Hg for each (b, wg, head)
    qc = Q.permute(0, 2, 3, 1, 4)
    O_ref, L_ref = oracle_mod.attention(qc, K.permute(0, 2, 3, 1, 4), V.permute(0, 2, 3, 1, 4), w.scale)
    assert_close(O_col.permute(0, 2, 3, 1, 4).cpu().numpy(), L_col.permute(0, 2, 3, 1).cpu().numpy(),
                 O_ref, L_ref, torch.float32, "axial col")


def sampled_rows(w, n_random=192, seed=7):
    """(b, h, rows) samples: the first and last 256 rows of the first and last
    (b, h) slice, plus random rows of random slices."""
    g = np.random.default_rng(seed)
    edge = sorted(set(list(range(min(256, w.N_q))) + list(range(max(0, w.N_q - 256), w.N_q))))
    out = [(0, 0, edge), (w.B - 1, w.H - 1, edge)]
    for _ in range(4):
        b, h = int(g.integers(w.B)), int(g.integers(w.H))
        out.append((b, h, sorted(g.choice(w.N_q, n_random // 4, replace=False).tolist())))
    return out


@pytest.mark.parametrize("name", ["large_nc", "large_causal", "cross_long_nc", "long_causal", "large_d64_nc",
                                  "large_d64_causal"])
def test_config_large_sampled(oracle_mod, name):
    """Full-size configurations in the launch configuration the benchmark times,
    checked on sampled rows against the oracle, plus properties on every row."""
    w = WORKLOADS[name]
    Q, K, V = w.make()
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    O = _poisoned(Q.shape, w.dtype)
    L = _poisoned(Q.shape[:-1], torch.float32)
    fa.fwd(Qd, Kd, Vd, scale=w.scale, is_causal=w.causal, out=O, lse=L)
    fa.check()
    assert bool(torch.isfinite(O).all()) and bool(torch.isfinite(L).all())
    # convex hull: every output lies within the range of V (per slice and column)
    vmax = Vd.float().amax(dim=2, keepdim=True)
    vmin = Vd.float().amin(dim=2, keepdim=True)
    assert bool((O.float() <= vmax + 2e-2).all()) and bool((O.float() >= vmin - 2e-2).all())
    worst = (0.0, 0.0)
    for b, h, rows in sampled_rows(w):
        O_ref, L_ref = oracle_mod.attention(Q[b, h], K[b, h], V[b, h], w.scale, w.causal, rows=rows)
        eo, el = assert_close(O[b, h, rows].float().cpu().numpy(), L[b, h, rows].cpu().numpy(),
                              O_ref, L_ref, w.dtype, f"{name} b={b} h={h}")
        worst = (max(worst[0], eo), max(worst[1], el))
    print(f"{name}: worst sampled max|dO|={worst[0]:.3e} max|dLSE|={worst[1]:.3e}")


# ------------------------------------------------------------- bounded waits
def test_withheld_tile_times_out_and_context_survives(oracle_mod):
    """The test hook withholds one K tile in block 0: the MMA warp's bounded
    wait runs out, the launch ends, fa_check reports FA_ERR_TIMEOUT, and the
    next launch on the same context is correct."""
    Q, K, V = (x.cuda() for x in qkv((1, 1, 512, 128), (1, 1, 512, 128), 81, torch.bfloat16))
    fa.debug_set(50_000_000, 1)  # 50 ms wait limit, withhold a tile
    try:
        fa.fwd(Q, K, V)
        with pytest.raises(fa.FaError) as ei:
            fa.check()
        assert ei.value.status == fa.FA_ERR_TIMEOUT
    finally:
        fa.debug_set(0, 0)
    fa.check()  # the error word was cleared
    Qh, Kh, Vh = (x.cpu() for x in (Q, K, V))
    O, L = run_gpu(Qh, Kh, Vh, 1 / math.sqrt(128), False)
    O_ref, L_ref = oracle_mod.attention(Qh, Kh, Vh, 1 / math.sqrt(128), False)
    assert_close(O, L, O_ref, L_ref, torch.bfloat16, "after timeout")
