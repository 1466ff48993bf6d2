"""Host-side logic of the benchmark and the input generators, on the CPU: the
workload registry, the FLOP and byte counts the roofline divides by, the
packed-batch offsets, and the determinism of the seeded inputs (the GPU path
and the oracle must read exactly the same numbers)."""
from __future__ import annotations

import json
import math

import numpy as np
import pytest
import torch

import bench
from attention_fa2_fwd_02_gb300.inputs import (AXIAL, AXIAL_BLOCK, VARLEN, WORKLOADS, VarlenWorkload, normal, packed,
                                               qkv, seq_lengths)


def test_every_workload_name_resolves():
    for name in list(WORKLOADS) + list(VARLEN) + ["axial", "axial_block"]:
        assert bench.get_workload(name) is not None
    for name in ("large_nc_bwd", "large_causal_bwd", "cross_long_nc_bwd", "large_d96_nc_bwd"):
        assert bench.get_workload(name) is WORKLOADS[name[:-4]]
    with pytest.raises(SystemExit):
        bench.get_workload("no_such_workload")
    with pytest.raises(SystemExit):
        bench.get_workload("tutorial_nc_bwd")  # the backward takes bf16 inputs only


def test_flops_count_both_products():
    # 2 N_q N_k d for Q K^T plus 2 N_q N_k Dv for P V, per (b, h); half under the causal mask
    for w in WORKLOADS.values():
        want = 2.0 * w.B * w.H * w.N_q * w.N_k * (w.d + w.v_dim) * (0.5 if w.causal else 1.0)
        assert w.flops == pytest.approx(want, rel=1e-15)
    big = WORKLOADS["large_nc"]
    assert big.flops == 4.0 * 4 * 32 * 8192 * 8192 * 128  # the pages' 4 z h n^2 d
    dv = WORKLOADS["large_dv64_nc"]
    assert dv.flops == pytest.approx(big.flops * (128 + 64) / 256)


def test_algorithmic_bytes():
    w = WORKLOADS["large_gqa_nc"]  # Q, O with 32 heads; K, V with 8
    e = 2
    want = (w.B * w.H * w.N_q * (w.d + w.v_dim) * e + w.B * w.kv_heads * w.N_k * (w.d + w.v_dim) * e
            + w.B * w.H * w.N_q * 4)
    assert w.algorithmic_bytes == want
    v = VARLEN["varlen_mix"]
    T = sum(v.lens)
    assert v.algorithmic_bytes == 2 * T * v.H * v.d * 2 + 2 * T * v.kv_heads * v.d * 2 + v.H * T * 4


def test_varlen_workload_counts():
    v = VARLEN["varlen_mix_causal"]
    assert v.flops == pytest.approx(sum(2.0 * v.H * v.d * n * n for n in v.lens))
    assert len(v.lens) == v.n_seq and all(v.lo <= n <= v.hi for n in v.lens)
    assert v.lens == VARLEN["varlen_mix"].lens  # same seed, same lengths
    desc = bench.workload_desc(v)
    assert desc["lengths"] == v.lens and "packed batch of 16 sequences" in desc["workload"]
    json.dumps(desc)


def test_packed_offsets_and_shapes():
    q, k, v, cu_q, cu_k = packed([3, 0, 5], [4, 2, 0], 6, 2, 16, seed=9)
    assert cu_q.tolist() == [0, 3, 3, 8] and cu_k.tolist() == [0, 4, 6, 6]
    assert cu_q.dtype == torch.int32 and cu_k.dtype == torch.int32
    assert q.shape == (8, 6, 16) and k.shape == (6, 2, 16) and v.shape == (6, 2, 16)
    assert q.dtype == torch.bfloat16
    q2, k2, v2, _, _ = packed([3, 0, 5], [4, 2, 0], 6, 2, 16, seed=9)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)


def test_seeded_inputs_are_deterministic_and_distinct():
    a = normal((4, 5), 7)
    assert torch.equal(a, normal((4, 5), 7))
    assert not torch.equal(a, normal((4, 5), 8))
    Q, K, V = qkv((2, 3, 4), (2, 5, 4), 11)
    assert not torch.equal(K, V)
    assert seq_lengths(10, 5, 9, 3) == seq_lengths(10, 5, 9, 3)
    # bf16 rounding of the same draw: what the GPU and the oracle both read
    b = normal((64,), 12, torch.bfloat16)
    assert torch.equal(b, normal((64,), 12).to(torch.bfloat16))


def test_value_dim_workload_inputs():
    Q, K, V = WORKLOADS["large_dv64_nc"].__class__(
        "t", 1, 2, 8, 9, 32, torch.bfloat16, False, 0.1, 5, 0, 16).make()
    assert Q.shape == (1, 2, 8, 32) and K.shape == (1, 2, 9, 32) and V.shape == (1, 2, 9, 16)


def test_axial_counts():
    assert AXIAL.flops > 0 and AXIAL.algorithmic_bytes > 0
    assert AXIAL_BLOCK.flops > 0 and AXIAL_BLOCK.algorithmic_bytes > 0
    assert math.isclose(AXIAL.scale, 0.25)


def test_whole_job_value_and_roofline_inputs():
    # value = FLOPs of all ranks / the slowest rank's step time
    assert bench.whole_job_value(2.0e12, 4, 2.0) == pytest.approx(4 * 2.0e12 / 2.0e-3 / 1e12)
    peaks, src = bench.load_peaks()
    assert float(peaks["bf16_tflops"]) > 0 and float(peaks["hbm_gbs"]) > 0 and src in ("measured", "fallback")


def test_recorded_traffic_matches_its_own_source_hash(tmp_path, monkeypatch):
    # a traffic record is reported only for the kernel sources it was taken on
    rec = {"source_hash": bench.kernel_source_hash(), "workloads": {"large_nc": {"dram_bytes_per_launch": 123.0}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["source_hash"])
    assert bench.recorded_traffic("large_nc") == 123.0
    assert bench.recorded_traffic("large_causal") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "other")
    assert bench.recorded_traffic("large_nc") is None


def test_numpy_float_inputs_for_the_oracle_are_exact():
    # every bf16 value widens exactly to fp32, so the oracle reads the GPU's inputs
    x = normal((1000,), 21, torch.bfloat16)
    assert np.array_equal(x.float().numpy().astype(np.float64), x.double().numpy())
    assert isinstance(VarlenWorkload, type)


def test_backward_flops():
    # five products: S, dK, dQ over d and dP, dV over Dv; 2.5x the forward when Dv = d
    big = WORKLOADS["large_nc"]
    assert bench.bwd_flops(big) == pytest.approx(2.5 * big.flops)
    dv = WORKLOADS["large_dv64_nc"]
    assert bench.bwd_flops(dv) == pytest.approx(2.0 * 4 * 32 * 8192 * 8192 * (3 * 128 + 2 * 64))
    assert bench.bwd_flops(WORKLOADS["large_causal"]) == pytest.approx(2.5 * WORKLOADS["large_causal"].flops)
