// fa_small.cuh -- FlashAttention-2 forward for small head dims (d = 16, 32)
// on the CUDA cores, for batches of short sequences such as the row and column
// attention of the axial-attention transcript (x[B, H, W, heads, hd] with
// hd = 16 and sequences of 32 along W or along H, scale = hd^-1/2).
//
// At d = 16 a score costs 16 multiply-adds and a tensor-core tile would be
// mostly padding; the work is dominated by moving Q, K, V and O, so the kernel
// is built around memory access instead:
//  * one warp owns 32 query rows of one (problem, b, h); lane = query row,
//    so the row max and row sum of the softmax stay inside a thread;
//  * K and V arrive 32 keys at a time, staged through shared memory with
//    coalesced 16-byte loads straight from the strided views (no copies of
//    the permuted column view are made), then read as warp-wide broadcasts;
//  * the online softmax (running max m and sum l, rescale by 2^(m_old-m_new))
//    of "Extend Thunder with CUDA-Python" (flash_attention_reference) makes
//    any N_k work; log2(e) is folded into the scale as in "Blackwell
//    Attention Example";
//  * O is staged through the same shared buffer and leaves with coalesced
//    16-byte stores; LSE (natural log) is written per row.
// Several problems run in one launch (work items are numbered across them).
#pragma once

#include "fa_ptx.cuh"

namespace fa {

constexpr int kSmallMaxGroup = 8;

struct SmallProblem {
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  float* LSE;
  long long qs[3], ks[3], vs[3], os[3], ls[3];  // element strides b, h, n
  int B, H, N_q, N_k;
  int kv_group;        // query heads per K/V head (grouped-query attention; 1 = none)
  int causal;
  int causal_off;      // causal: key j visible to row i iff j <= i + causal_off
  float scale_log2;
  int n_qblk;          // ceil(N_q / 32)
  int vec_ok;          // every row starts on a 16-byte boundary
  long long item_begin;
};

struct SmallParams {
  int n_problems;
  long long n_items;
  SmallProblem prob[kSmallMaxGroup];
};

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Stage rows [r0, r0+32) x D of a strided [N, D] view into dst[32][D+4]
// (fp32); rows at or past n_rows read as zero.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(float* dst, const T* base, long long rs, int r0, int n_rows,
                                           bool vec, int lane) {
  constexpr int LD = D + 4;
  if (vec) {
    constexpr int V = 16 / sizeof(T);        // elements per 16-byte vector
    constexpr int VPR = D / V;               // vectors per row
    constexpr int TOTAL = 32 * VPR;
#pragma unroll
    for (int idx = lane; idx < TOTAL; idx += 32) {
      const int r = idx / VPR, cv = idx % VPR;
      float* d = dst + r * LD + cv * V;
      if (r0 + r < n_rows) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + (long long)(r0 + r) * rs + cv * V);
        if constexpr (sizeof(T) == 4) {
          *reinterpret_cast<float4*>(d) = make_float4(__uint_as_float(w.x), __uint_as_float(w.y),
                                                      __uint_as_float(w.z), __uint_as_float(w.w));
        } else {
          const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            d[2 * k] = __uint_as_float(u[k] << 16);
            d[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < V; ++k) d[k] = 0.f;
      }
    }
  } else {
    for (int idx = lane; idx < 32 * D; idx += 32) {
      const int r = idx / D, c = idx % D;
      dst[r * LD + c] = (r0 + r < n_rows) ? to_f32<T>(base[(long long)(r0 + r) * rs + c]) : 0.f;
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(128)
fa_small_fwd_kernel(const __grid_constant__ SmallParams P) {
  constexpr int LD = D + 4;
  extern __shared__ float small_smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  float* sQ = small_smem + warp * (3 * 32 * LD);  // Q, later O
  float* sK = sQ + 32 * LD;
  float* sV = sK + 32 * LD;

  const long long item = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (item >= P.n_items) return;
  int pi = 0;
#pragma unroll 1
  while (pi + 1 < P.n_problems && item >= P.prob[pi + 1].item_begin) ++pi;
  const SmallProblem& pr = P.prob[pi];
  long long rem = item - pr.item_begin;
  const int qb = static_cast<int>(rem % pr.n_qblk);
  rem /= pr.n_qblk;
  const int h = static_cast<int>(rem % pr.H);
  const int b = static_cast<int>(rem / pr.H);
  const int r0 = qb * 32;
  const int q = r0 + lane;
  const bool vec = pr.vec_ok != 0;

  const T* Qb = reinterpret_cast<const T*>(pr.Q) + b * pr.qs[0] + h * pr.qs[1];
  const int hk = h / pr.kv_group;  // the K/V head of query head h
  const T* Kb = reinterpret_cast<const T*>(pr.K) + b * pr.ks[0] + hk * pr.ks[1];
  const T* Vb = reinterpret_cast<const T*>(pr.V) + b * pr.vs[0] + hk * pr.vs[1];

  stage_rows<T, D>(sQ, Qb, pr.qs[2], r0, pr.N_q, vec, lane);
  __syncwarp();
  float qr[D];
#pragma unroll
  for (int c = 0; c < D; c += 4) {
    const float4 v = *reinterpret_cast<const float4*>(sQ + lane * LD + c);
    qr[c] = v.x * pr.scale_log2;
    qr[c + 1] = v.y * pr.scale_log2;
    qr[c + 2] = v.z * pr.scale_log2;
    qr[c + 3] = v.w * pr.scale_log2;
  }
  float acc[D];
#pragma unroll
  for (int c = 0; c < D; ++c) acc[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int vis_end = pr.causal ? min(pr.N_k, q + 1 + pr.causal_off) : pr.N_k;   // this lane's keys
  const int kv_end = pr.causal ? min(pr.N_k, r0 + 32 + pr.causal_off) : pr.N_k;  // the warp's keys

#pragma unroll 1
  for (int kc = 0; kc < kv_end; kc += 32) {
    __syncwarp();
    stage_rows<T, D>(sK, Kb, pr.ks[2], kc, pr.N_k, vec, lane);
    stage_rows<T, D>(sV, Vb, pr.vs[2], kc, pr.N_k, vec, lane);
    __syncwarp();
    float s[32];
    float mloc = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < D; c += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(sK + jj * LD + c);
        dot = fmaf(qr[c], k4.x, dot);
        dot = fmaf(qr[c + 1], k4.y, dot);
        dot = fmaf(qr[c + 2], k4.z, dot);
        dot = fmaf(qr[c + 3], k4.w, dot);
      }
      s[jj] = (kc + jj < vis_end) ? dot : -INFINITY;
      mloc = fmaxf(mloc, s[jj]);
    }
    const float m_new = fmaxf(m, mloc);
    // m = -inf on the first chunk -> 0; a row that has seen no key keeps 1
    const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
    l *= alpha;
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] *= alpha;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const float p = (kc + jj < vis_end) ? ex2(s[jj] - m_new) : 0.f;
      l += p;
#pragma unroll
      for (int c = 0; c < D; c += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(sV + jj * LD + c);
        acc[c] = fmaf(p, v4.x, acc[c]);
        acc[c + 1] = fmaf(p, v4.y, acc[c + 1]);
        acc[c + 2] = fmaf(p, v4.z, acc[c + 2]);
        acc[c + 3] = fmaf(p, v4.w, acc[c + 3]);
      }
    }
    m = m_new;
  }

  // epilogue: O = acc / l through shared memory, LSE = (m + log2 l) ln 2
  const float inv = l > 0.f ? 1.f / l : 0.f;  // a row that sees no key: O = 0, LSE = -inf
  __syncwarp();
#pragma unroll
  for (int c = 0; c < D; c += 4)
    *reinterpret_cast<float4*>(sQ + lane * LD + c) =
        make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
  __syncwarp();
  T* Ob = reinterpret_cast<T*>(pr.O) + b * pr.os[0] + h * pr.os[1];
  if (vec) {
    constexpr int V = 16 / sizeof(T);
    constexpr int VPR = D / V;
#pragma unroll
    for (int idx = lane; idx < 32 * VPR; idx += 32) {
      const int r = idx / VPR, cv = idx % VPR;
      if (r0 + r >= pr.N_q) continue;
      const float* src = sQ + r * LD + cv * V;
      uint4 w;
      if constexpr (sizeof(T) == 4) {
        w = make_uint4(__float_as_uint(src[0]), __float_as_uint(src[1]), __float_as_uint(src[2]),
                       __float_as_uint(src[3]));
      } else {
        w = make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]),
                       pack_bf16x2(src[4], src[5]), pack_bf16x2(src[6], src[7]));
      }
      *reinterpret_cast<uint4*>(Ob + (long long)(r0 + r) * pr.os[2] + cv * V) = w;
    }
  } else {
    for (int idx = lane; idx < 32 * D; idx += 32) {
      const int r = idx / D, c = idx % D;
      if (r0 + r >= pr.N_q) continue;
      const float v = sQ[r * LD + c];
      T* dst = Ob + (long long)(r0 + r) * pr.os[2] + c;
      if constexpr (sizeof(T) == 4) {
        *dst = v;
      } else {
        *dst = __float2bfloat16_rn(v);
      }
    }
  }
  if (q < pr.N_q && pr.LSE)
    pr.LSE[b * pr.ls[0] + h * pr.ls[1] + (long long)q * pr.ls[2]] = (m + __log2f(l)) * 0.69314718055994531f;
}

template <typename T, int D>
constexpr int small_smem_bytes() {
  return 4 * 3 * 32 * (D + 4) * static_cast<int>(sizeof(float));
}

}  // namespace fa
