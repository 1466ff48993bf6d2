"""Seeded synthetic inputs and the workload shapes.

This module is shared by the tests, the benchmark and the smoke check.  It
holds no attention arithmetic: it only draws i.i.d. N(0, 1) values from a
seeded CPU generator and rounds them to the storage dtype, so that the GPU
path and the fp64 oracle read exactly the same numbers.

The workloads mirror the pages' own inputs, which are all ``torch.randn``
draws: the 96 x 512 x 128 fp32 batch of "Extend Thunder with CUDA-Python"
(opening section), the (4, 32, 8192, {64,128}) bf16 shapes of "Blackwell
Attention Example" (section "Main Function"), and the axial grid of the
axial-attention transcript (B=4, H=W=32, 4 heads of dim 16).
"""
from __future__ import annotations

import math
import itertools
from dataclasses import dataclass

import torch


def normal(shape, seed: int, dtype=torch.float32) -> torch.Tensor:
    """i.i.d. N(0,1) on the CPU from a seeded generator, rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    return x.to(dtype)


def qkv(q_shape, kv_shape, seed: int, dtype=torch.float32):
    """Q, K, V drawn with seeds 3*seed, 3*seed+1, 3*seed+2."""
    return (normal(q_shape, 3 * seed, dtype),
            normal(kv_shape, 3 * seed + 1, dtype),
            normal(kv_shape, 3 * seed + 2, dtype))


def packed(lens_q, lens_k, H: int, H_kv: int, d: int, seed: int, dtype=torch.bfloat16):
    """A packed variable-length batch: q [sum lens_q, H, d], k and v
    [sum lens_k, H_kv, d] (N(0,1), seeded), and the int32 offsets
    cu_q = [0, cumsum(lens_q)], cu_k = [0, cumsum(lens_k)] (CPU tensors)."""
    cu_q = torch.tensor([0] + list(itertools.accumulate(int(n) for n in lens_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(int(n) for n in lens_k)), dtype=torch.int32)
    q, k, v = (normal((int(cu_q[-1]), H, d), 3 * seed, dtype),
               normal((int(cu_k[-1]), H_kv, d), 3 * seed + 1, dtype),
               normal((int(cu_k[-1]), H_kv, d), 3 * seed + 2, dtype))
    return q, k, v, cu_q, cu_k


def seq_lengths(n: int, lo: int, hi: int, seed: int):
    """n sequence lengths drawn uniformly from [lo, hi] with a seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


@dataclass(frozen=True)
class Workload:
    """One attention problem in the SDPA layout [B, H, N, d]."""
    name: str
    B: int
    H: int
    N_q: int
    N_k: int
    d: int
    dtype: torch.dtype
    causal: bool
    scale: float
    seed: int
    H_kv: int = 0  # K/V heads (grouped-query attention); 0 = H
    Dv: int = 0    # head dim of V and O; 0 = d

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def v_dim(self) -> int:
        return self.Dv or self.d

    @property
    def flops(self) -> float:
        """2 * B * H * N_q * N_k * (d + Dv) (Q K^T and P V; 4 B H N_q N_k d
        when Dv = d), halved for causal attention."""
        f = 2.0 * self.B * self.H * self.N_q * self.N_k * (self.d + self.v_dim)
        return f / 2 if self.causal else f

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == torch.bfloat16 else 4

    @property
    def algorithmic_bytes(self) -> float:
        """Q, K, V read once; O written once (input dtype); LSE written (fp32)."""
        e = self.elem_bytes
        q = self.B * self.H * self.N_q * self.d * e
        kv = self.B * self.kv_heads * self.N_k * (self.d + self.v_dim) * e
        o = self.B * self.H * self.N_q * self.v_dim * e
        lse = self.B * self.H * self.N_q * 4
        return float(q + kv + o + lse)

    def make(self):
        Q, K, V = qkv((self.B, self.H, self.N_q, self.d),
                      (self.B, self.kv_heads, self.N_k, self.d), self.seed, self.dtype)
        if self.v_dim != self.d:
            V = normal((self.B, self.kv_heads, self.N_k, self.v_dim), 3 * self.seed + 2, self.dtype)
        return Q, K, V


def _w(name, B, H, Nq, Nk, d, dtype, causal, scale=None, seed=0, H_kv=0, Dv=0):
    return Workload(name, B, H, Nq, Nk, d, dtype, causal,
                    1.0 / math.sqrt(d) if scale is None else scale, seed, H_kv, Dv)


# The five configurations (non-causal and causal variants where both are run).
WORKLOADS = {
    "tiny_nc": _w("tiny_nc", 1, 1, 64, 64, 64, torch.float32, False, seed=1),
    "tiny_causal": _w("tiny_causal", 1, 1, 64, 64, 64, torch.float32, True, seed=1),
    "tutorial_nc": _w("tutorial_nc", 96, 1, 512, 512, 128, torch.float32, False, seed=2),
    "tutorial_causal": _w("tutorial_causal", 96, 1, 512, 512, 128, torch.float32, True, seed=2),
    "large_nc": _w("large_nc", 4, 32, 8192, 8192, 128, torch.bfloat16, False, seed=4),
    "large_causal": _w("large_causal", 4, 32, 8192, 8192, 128, torch.bfloat16, True, seed=4),
    "cross_long_nc": _w("cross_long_nc", 2, 16, 4096, 32768, 64, torch.bfloat16, False, seed=5),
    "long_causal": _w("long_causal", 1, 16, 32768, 32768, 128, torch.bfloat16, True, seed=6),
    # grouped-query attention: the large self-attention shape with 8 K/V heads
    "large_gqa_nc": _w("large_gqa_nc", 4, 32, 8192, 8192, 128, torch.bfloat16, False, seed=9, H_kv=8),
    "large_gqa_causal": _w("large_gqa_causal", 4, 32, 8192, 8192, 128, torch.bfloat16, True, seed=9, H_kv=8),
    # other head dims: d = 96 (computed on 128-column tiles), and V with 64
    # columns against d = 128
    "large_d96_nc": _w("large_d96_nc", 4, 32, 8192, 8192, 96, torch.bfloat16, False, seed=10),
    "large_d96_causal": _w("large_d96_causal", 4, 32, 8192, 8192, 96, torch.bfloat16, True, seed=10),
    "large_dv64_nc": _w("large_dv64_nc", 4, 32, 8192, 8192, 128, torch.bfloat16, False, seed=11, Dv=64),
    # head dim 64 at the large shape ("Blackwell Attention Example", main():
    # (4, 32, 8192, 64) bf16)
    "large_d64_nc": _w("large_d64_nc", 4, 32, 8192, 8192, 64, torch.bfloat16, False, seed=14),
    "large_d64_causal": _w("large_d64_causal", 4, 32, 8192, 8192, 64, torch.bfloat16, True, seed=14),
    # head dim 256 (the single-stage kernel for head dims above 128)
    "large_d256_nc": _w("large_d256_nc", 4, 32, 8192, 8192, 256, torch.bfloat16, False, seed=12),
    "large_d256_causal": _w("large_d256_causal", 4, 32, 8192, 8192, 256, torch.bfloat16, True, seed=12),
    # profiling-size cases of the same kernels: inputs still larger than the
    # 129 MB L2, but small enough for a many-pass ncu capture
    "prof_nc": _w("prof_nc", 1, 32, 8192, 8192, 128, torch.bfloat16, False, seed=7),
    "prof_causal": _w("prof_causal", 1, 32, 8192, 8192, 128, torch.bfloat16, True, seed=7),
    "prof_cross": _w("prof_cross", 1, 16, 4096, 32768, 64, torch.bfloat16, False, seed=8),
    "prof_tutorial": _w("prof_tutorial", 96, 1, 512, 512, 128, torch.float32, False, seed=2),
    "prof_d256_nc": _w("prof_d256_nc", 1, 32, 8192, 8192, 256, torch.bfloat16, False, seed=13),
}


@dataclass(frozen=True)
class AxialWorkload:
    """Axial attention core over a grid x[B, Hg, Wg, heads, hd] (fp32).

    Row attention: sequences of length Wg, one per (b, hg, head).
    Column attention: sequences of length Hg, one per (b, wg, head).
    Both read Q, K, V of shape [B, Hg, Wg, heads, hd] in place (strided).
    """
    name: str = "axial"
    B: int = 4
    Hg: int = 32
    Wg: int = 32
    heads: int = 4
    hd: int = 16
    scale: float = 0.25
    seed: int = 3

    @property
    def shape(self):
        return (self.B, self.Hg, self.Wg, self.heads, self.hd)

    @property
    def flops(self) -> float:
        """Row plus column attention: 4 * (#sequences) * L^2 * hd each."""
        row = 4.0 * self.B * self.Hg * self.heads * self.Wg * self.Wg * self.hd
        col = 4.0 * self.B * self.Wg * self.heads * self.Hg * self.Hg * self.hd
        return row + col

    @property
    def algorithmic_bytes(self) -> float:
        """Per direction: Q, K, V read, O written (fp32), LSE written (fp32)."""
        n = self.B * self.Hg * self.Wg * self.heads
        per_dir = 4 * n * self.hd * 4 + n * 4
        return 2.0 * per_dir

    def make(self):
        return qkv(self.shape, self.shape, self.seed, torch.float32)


AXIAL = AxialWorkload()


@dataclass(frozen=True)
class AxialBlockWorkload:
    """The whole axial attention block (row pass then column pass) on a grid
    x [B, H, W, D] fp32 with random weights: LayerNorm, QKV projection,
    4-head attention, output projection with bias, residual, per pass."""
    name: str = "axial_block"
    B: int = 4
    H: int = 32
    W: int = 32
    D: int = 64
    heads: int = 4
    seed: int = 11

    @property
    def shape(self):
        return (self.B, self.H, self.W, self.D)

    @property
    def flops(self) -> float:
        """Per pass and sequence of L tokens: QKV 2*L*D*3D, attention
        4*L^2*D, output projection 2*L*D*D (LayerNorm, softmax and the
        residual not counted)."""
        def per_seq(L):
            return 2.0 * L * self.D * 3 * self.D + 4.0 * L * L * self.D + 2.0 * L * self.D * self.D
        return self.B * self.H * per_seq(self.W) + self.B * self.W * per_seq(self.H)

    @property
    def algorithmic_bytes(self) -> float:
        """The grid read and written once per pass, both passes' weights read once."""
        grid = self.B * self.H * self.W * self.D * 4
        weights = 2 * (3 * self.D * self.D + self.D * self.D + 3 * self.D) * 4
        return 4.0 * grid + weights

    def weights(self, seed):
        D = self.D
        return dict(norm_w=1.0 + 0.1 * normal((D,), seed), norm_b=0.1 * normal((D,), seed + 1),
                    qkv_w=normal((3 * D, D), seed + 2) / 8.0, out_w=normal((D, D), seed + 3) / 8.0,
                    out_b=0.1 * normal((D,), seed + 4))

    def make(self):
        """x, row weights, column weights (CPU fp32; weights ~ nn.Linear scale 1/sqrt(D))."""
        return normal(self.shape, 3 * self.seed), self.weights(10 * self.seed), self.weights(10 * self.seed + 5)


AXIAL_BLOCK = AxialBlockWorkload()


@dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of self-attention sequences of mixed lengths (a training
    batch of packed documents): n_seq lengths drawn uniformly from [lo, hi]
    with a seeded generator, H heads of dim d, bf16, N(0, 1) inputs."""
    name: str
    n_seq: int
    lo: int
    hi: int
    H: int
    d: int
    causal: bool
    seed: int
    H_kv: int = 0

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def lens(self):
        return seq_lengths(self.n_seq, self.lo, self.hi, self.seed)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4 H d L^2 per sequence (two matmuls), halved under the causal mask."""
        f = sum(4.0 * self.H * self.d * n * n for n in self.lens)
        return f / 2 if self.causal else f

    @property
    def algorithmic_bytes(self) -> float:
        """q, k, v read once; O written once (bf16); LSE written (fp32)."""
        T = sum(self.lens)
        return float(2 * T * self.H * self.d * 2 + 2 * T * self.kv_heads * self.d * 2 + self.H * T * 4)

    def make(self):
        return packed(self.lens, self.lens, self.H, self.kv_heads, self.d, self.seed, torch.bfloat16)


VARLEN = {
    "varlen_mix": VarlenWorkload("varlen_mix", 16, 512, 8192, 32, 128, False, seed=31),
    "varlen_mix_causal": VarlenWorkload("varlen_mix_causal", 16, 512, 8192, 32, 128, True, seed=31),
}
