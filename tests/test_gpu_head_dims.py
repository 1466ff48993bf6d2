"""Head dims other than 64 and 128, and V with a head dim of its own
("Blackwell Attention Example", blackwell_attention: Q and K share d, V and O
have Dv columns), on the tensor-core path, against the oracle element by
element.

The tiles are 64, 128 or (bf16, the single-stage kernel for head dims above
128) 256 columns wide; a smaller d or Dv is computed on tiles whose extra
columns are loaded as zeros.  Every case writes O into a view of a wider
buffer whose extra columns hold NaN, so a store past Dv is caught."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import attention_fa2_fwd_02_gb300 as fa
from attention_fa2_fwd_02_gb300.inputs import normal, packed, qkv

pytestmark = pytest.mark.gpu
TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float32: (3e-3, 2e-3)}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa.build()
    fa.debug_set(0, 0)
    yield


def _run(oracle_mod, dtype, d, dv, causal, B=2, H=3, H_kv=None, nq=300, nk=300, seed=0, via="fwd"):
    H_kv = H_kv or H
    Q, K, _ = qkv((B, H, nq, d), (B, H_kv, nk, d), 2000 + seed, dtype)
    V = normal((B, H_kv, nk, dv), 2100 + seed, dtype)
    scale = 1.0 / math.sqrt(d)
    pad = 16 // torch.empty((), dtype=dtype).element_size()  # extra columns: one 16-byte group
    buf = torch.full((B, H, nq, dv + pad), float("nan"), dtype=dtype, device="cuda")
    O = buf[..., :dv]
    L = torch.full((B, H, nq), float("nan"), dtype=torch.float32, device="cuda")
    if via == "fwd":
        fa.fwd(Q.cuda(), K.cuda(), V.cuda(), scale=scale, is_causal=causal, out=O, lse=L)
    else:
        fa.fwd_noalloc(Q.cuda(), K.cuda(), V.cuda(), out=O, lse=L, scale=scale, is_causal=causal)
    fa.check()
    G = H // H_kv
    O_ref, L_ref = oracle_mod.attention(Q, K.repeat_interleave(G, 1), V.repeat_interleave(G, 1), scale,
                                        fa.causal_code(causal))
    assert torch.isnan(buf[..., dv:]).all(), "a column past Dv was written"
    to, tl = TOL[dtype]
    Og, Lg = O.float().cpu().numpy(), L.cpu().numpy()
    fin = np.isfinite(L_ref)
    assert np.array_equal(np.isneginf(Lg), np.isneginf(L_ref))
    eo = float(np.abs(Og - O_ref).max())
    el = float(np.abs(Lg[fin] - L_ref[fin]).max(initial=0.0))
    assert eo <= to and el <= tl, f"max|dO|={eo:.3e} max|dLSE|={el:.3e}"


@pytest.mark.parametrize("d", [8, 24, 40, 48, 80, 96, 112])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"], ids=["nc", "top_left", "bottom_right"])
def test_bf16_head_dims(oracle_mod, d, causal):
    _run(oracle_mod, torch.bfloat16, d, d, causal, nq=300, nk=333 if causal != "bottom_right" else 200, seed=d)


@pytest.mark.parametrize("d,dv", [(64, 128), (128, 64), (96, 64), (32, 128), (16, 64), (128, 8), (64, 32),
                                  (40, 104)])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bf16_value_dim(oracle_mod, d, dv, causal):
    _run(oracle_mod, torch.bfloat16, d, dv, causal, nq=257, nk=385, seed=d + dv)


@pytest.mark.parametrize("d,dv", [(20, 20), (44, 44), (96, 96), (64, 32), (128, 36)])
@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_fp32_head_dims(oracle_mod, d, dv, causal):
    _run(oracle_mod, torch.float32, d, dv, causal, nq=200, nk=150, seed=3 * d + dv)


@pytest.mark.parametrize("H,H_kv", [(6, 2), (4, 1)])
def test_value_dim_with_grouped_heads(oracle_mod, H, H_kv):
    _run(oracle_mod, torch.bfloat16, 128, 64, True, H=H, H_kv=H_kv, nq=300, nk=300, seed=H + H_kv)
    _run(oracle_mod, torch.bfloat16, 96, 96, False, H=H, H_kv=H_kv, nq=129, nk=500, seed=7 + H_kv)


def test_value_dim_without_allocation(oracle_mod):
    _run(oracle_mod, torch.bfloat16, 128, 64, False, via="noalloc", seed=11)
    _run(oracle_mod, torch.bfloat16, 80, 80, True, via="noalloc", seed=12)


@pytest.mark.parametrize("d,dv", [(96, 96), (128, 64), (64, 112)])
def test_varlen_head_dims(oracle_mod, d, dv):
    lens_q, lens_k = [300, 0, 129, 513], [200, 7, 129, 600]
    q, k, _, cu_q, cu_k = packed(lens_q, lens_k, 4, 2, d, 2200 + d, torch.bfloat16)
    v = normal((k.shape[0], 2, dv), 2300 + dv, torch.bfloat16)
    O, L = fa.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), max(lens_q), is_causal=True)
    fa.check()
    assert O.shape == (q.shape[0], 4, dv)
    O_ref, L_ref = oracle_mod.attention_varlen(q.float().numpy(), k.float().repeat_interleave(2, 1).numpy(),
                                               v.float().repeat_interleave(2, 1).numpy(), cu_q.numpy(),
                                               cu_k.numpy(), 1.0 / math.sqrt(d), 1)
    assert float(np.abs(O.float().cpu().numpy() - O_ref).max()) <= 2e-2
    assert float(np.abs(L.cpu().numpy() - L_ref).max()) <= 1e-2


def test_sdpa_value_dim(oracle_mod):
    import torch.nn.functional as F

    from attention_fa2_fwd_02_gb300 import sdpa
    Q, K, _ = qkv((2, 4, 200, 128), (2, 4, 300, 128), 2400, torch.bfloat16)
    V = normal((2, 4, 300, 64), 2401, torch.bfloat16)
    with sdpa.routed():
        O = F.scaled_dot_product_attention(Q.cuda(), K.cuda(), V.cuda(), is_causal=True)
    fa.check()
    O_ref, _ = oracle_mod.attention(Q, K, V, 1.0 / math.sqrt(128), True)
    assert O.shape == (2, 4, 200, 64)
    assert float(np.abs(O.float().cpu().numpy() - O_ref).max()) <= 2e-2


@pytest.mark.parametrize("d,dv", [(256, 256), (192, 192), (136, 136), (192, 128), (256, 64), (64, 256),
                                  (128, 200)])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"], ids=["nc", "top_left", "bottom_right"])
def test_bf16_wide_head_dims(oracle_mod, d, dv, causal):
    # 128-row query blocks and 128-key tiles: 300 / 333 rows leave ragged tails on both
    _run(oracle_mod, torch.bfloat16, d, dv, causal, nq=300, nk=333 if causal != "bottom_right" else 200,
         seed=5 * d + dv)


@pytest.mark.parametrize("nq,nk", [(1, 1), (1, 700), (129, 128), (64, 129), (700, 1)])
def test_bf16_wide_edge_lengths(oracle_mod, nq, nk):
    for causal in (False, True, "bottom_right"):
        _run(oracle_mod, torch.bfloat16, 256, 256, causal, B=1, H=2, nq=nq, nk=nk, seed=nq + nk)


def test_bf16_wide_grouped_heads_and_noalloc(oracle_mod):
    _run(oracle_mod, torch.bfloat16, 256, 256, True, H=6, H_kv=2, nq=257, nk=257, seed=31)
    _run(oracle_mod, torch.bfloat16, 192, 128, False, H=4, H_kv=1, nq=200, nk=640, seed=32)
    _run(oracle_mod, torch.bfloat16, 256, 256, False, via="noalloc", seed=33)


def test_bf16_wide_many_tiles_sampled(oracle_mod):
    # more query blocks than SMs (persistent schedule) and long key ranges: sampled rows
    B, H, N, d = 2, 16, 2048, 256
    Q, K, V = qkv((B, H, N, d), (B, H, N, d), 2500, torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        O, L = fa.fwd(Q.cuda(), K.cuda(), V.cuda(), scale=scale, is_causal=causal)
        fa.check()
        rows = np.array([0, 1, 127, 128, 1000, 2047])
        for b, h in ((0, 0), (1, 15), (0, 7)):
            Or, Lr = oracle_mod.attention(Q[b, h], K[b, h], V[b, h], scale, causal, rows=rows)
            assert float(np.abs(O[b, h, rows].float().cpu().numpy() - Or).max()) <= 2e-2
            assert float(np.abs(L[b, h, rows].cpu().numpy() - Lr).max()) <= 1e-2


def test_unsupported_dims_raise():
    Q, K, V = (torch.zeros((1, 1, 64, n), dtype=torch.bfloat16, device="cuda") for n in (264, 264, 264))
    with pytest.raises(fa.FaError):
        fa.fwd(Q, K, V)                      # above the 256-column tile
    Q, K, V = (torch.zeros((1, 1, 64, 136), dtype=torch.float32, device="cuda") for _ in range(3))
    with pytest.raises(fa.FaError):
        fa.fwd(Q, K, V)                      # fp32 stops at 128
    Q, K, V = (torch.zeros((1, 1, 64, 100), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    with pytest.raises(fa.FaError):
        fa.fwd(Q, K, V)                      # a 200-byte row
    Q, K, V = (torch.zeros((1, 1, 64, 256), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    O, L = fa.fwd(Q, K, V)
    with pytest.raises(fa.FaError):
        fa.bwd(Q, K, V, O, L, O.clone())     # the backward stops at 128


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bf16_wide_strided_head_major(oracle_mod, causal):
    # Q, K, V, O as [B, H, N, d] views of [B, N, H, d] storage (no copies): the tensor maps take the strides
    B, H, N, d = 2, 3, 300, 256
    Q, K, V = qkv((B, H, N, d), (B, H, N, d), 2600, torch.bfloat16)
    dev = [x.transpose(1, 2).contiguous().cuda().transpose(1, 2) for x in (Q, K, V)]
    O = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    scale = 1.0 / math.sqrt(d)
    _, L = fa.fwd(*dev, scale=scale, is_causal=causal, out=O)
    fa.check()
    O_ref, L_ref = oracle_mod.attention(Q, K, V, scale, causal)
    assert float(np.abs(O.float().cpu().numpy() - O_ref).max()) <= 2e-2
    assert float(np.abs(L.cpu().numpy() - L_ref).max()) <= 1e-2
