// fa_small.cuh -- FlashAttention-2 forward for small head dims (d = 16, 32)
// on the CUDA cores, for batches of short sequences such as the row and column
// attention of the axial-attention transcript (x[B, H, W, heads, hd] with
// hd = 16 and sequences of 32 along W or along H, scale = hd^-1/2).
//
// At d = 16 a score costs 16 multiply-adds and a tensor-core tile would be
// mostly padding; the work is dominated by moving Q, K, V and O, and a launch
// of the axial shape moves about one memory round trip's worth of data, so the
// kernel is built around latency:
//  * one 128-thread CTA owns 32 query rows of one (problem, b, h); four
//    threads share a query row, each taking every fourth key of a 32-key
//    chunk (keys 4k + t), so that a thread's dependent chain is a quarter of
//    the row's work and the four rows of K or V read at once fall on distinct
//    banks;
//  * Q, K and V arrive 32 rows at a time, staged through shared memory with
//    coalesced 16-byte loads straight from the strided views (no copies of
//    the permuted column view are made); the loads of the Q block and of the
//    first K/V chunk are all issued before any of them is used (one memory
//    round trip), and the next chunk is loaded into registers while the
//    current one is computed;
//  * each thread keeps the online softmax (running max m, sum l, output
//    rescaled by 2^(m_old - m_new)) of "Extend Thunder with CUDA-Python"
//    (flash_attention_reference) over its keys, with log2(e) folded into the
//    scale as in "Blackwell Attention Example"; the four partial results of a
//    row are merged at the end with the same rescaling identity (warp
//    shuffles: M = max m_t, l = sum l_t 2^(m_t - M), O likewise);
//  * O is staged through shared memory and leaves with coalesced 16-byte
//    stores; LSE (natural log) is written per row.
// Several problems run in one launch (work items are numbered across them).
#pragma once

#include "fa_ptx.cuh"

namespace fa {

constexpr int kSmallMaxGroup = 8;
constexpr int kSmallSplit = 2;  // threads per query row of the launched kernel

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

// 32 rows x D of a row-aligned [N, D] view in registers, spread over the CTA:
// thread t holds the 16-byte vectors t, t + 128, ... of the chunk (row =
// index / vectors per row).
template <typename T, int D, int NT>
struct RowChunk {
  static constexpr int kVec = 16 / sizeof(T);            // elements per 16-byte vector
  static constexpr int kVpr = D / kVec;                  // vectors per row
  static constexpr int kTotal = 32 * kVpr;
  static constexpr int kPer = (kTotal + NT - 1) / NT;
  uint4 v[kPer];
};

// Rows [r0, r0 + 32); rows at or past n_rows read as zero.
template <typename T, int D, int NT>
__device__ __forceinline__ void load_chunk(RowChunk<T, D, NT>& c, const T* base, long long rs, int r0, int n_rows,
                                           int tid) {
  using C = RowChunk<T, D, NT>;
#pragma unroll
  for (int i = 0; i < C::kPer; ++i) {
    const int idx = tid + NT * i, r = idx / C::kVpr, cv = idx % C::kVpr;
    c.v[i] = (idx < C::kTotal && r0 + r < n_rows)
                 ? *reinterpret_cast<const uint4*>(base + (long long)(r0 + r) * rs + cv * C::kVec)
                 : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The chunk into dst[32][D+4] (fp32).
template <typename T, int D, int NT>
__device__ __forceinline__ void store_chunk(float* dst, const RowChunk<T, D, NT>& c, int tid) {
  using C = RowChunk<T, D, NT>;
  constexpr int LD = D + 4;
#pragma unroll
  for (int i = 0; i < C::kPer; ++i) {
    const int idx = tid + NT * i, r = idx / C::kVpr, cv = idx % C::kVpr;
    if (idx >= C::kTotal) break;
    float* d = dst + r * LD + cv * C::kVec;
    const uint4 w = c.v[i];
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
  }
}

// Rows [r0, r0+32) x D of a strided [N, D] view into dst[32][D+4] (fp32),
// element by element (views whose rows are not 16-byte aligned); rows at or
// past n_rows read as zero.
template <typename T, int D, int NT>
__device__ __forceinline__ void stage_rows_scalar(float* dst, const T* base, long long rs, int r0, int n_rows,
                                                  int tid) {
  constexpr int LD = D + 4;
  for (int idx = tid; idx < 32 * D; idx += NT) {
    const int r = idx / D, c = idx % D;
    dst[r * LD + c] = (r0 + r < n_rows) ? to_f32<T>(base[(long long)(r0 + r) * rs + c]) : 0.f;
  }
}

// kSplit threads per query row (1, 2 or 4): a CTA of 32 * kSplit threads.
template <typename T, int D, int kSplit>
__global__ void __launch_bounds__(32 * kSplit)
fa_small_fwd_kernel(const __grid_constant__ SmallParams P) {
  constexpr int kSmallThreads = 32 * kSplit;
  constexpr int kSmallSplit = kSplit;
  constexpr int LD = D + 4;  // shared row pitch: rows 4 floats apart in bank terms
  extern __shared__ float small_smem[];
  float* sQ = small_smem;    // Q, later O
  float* sK = sQ + 32 * LD;
  float* sV = sK + 32 * LD;
  const int tid = threadIdx.x;

  const long long item = static_cast<long long>(blockIdx.x);
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
  const int qi = tid / kSmallSplit;  // query row of the block
  const int kt = tid % kSmallSplit;  // this thread's keys: kt, kt + 4, ... of each chunk
  const int q = r0 + qi;
  const bool vec = pr.vec_ok != 0;

  const T* Qb = reinterpret_cast<const T*>(pr.Q) + b * pr.qs[0] + h * pr.qs[1];
  const int hk = h / pr.kv_group;  // the K/V head of query head h
  const T* Kb = reinterpret_cast<const T*>(pr.K) + b * pr.ks[0] + hk * pr.ks[1];
  const T* Vb = reinterpret_cast<const T*>(pr.V) + b * pr.vs[0] + hk * pr.vs[1];

  const int vis_end = pr.causal ? min(pr.N_k, q + 1 + pr.causal_off) : pr.N_k;   // this row's keys
  const int kv_end = pr.causal ? min(pr.N_k, r0 + 32 + pr.causal_off) : pr.N_k;  // the block's keys
  if (vec) {
    // Q, K and V of the first chunk: every load in flight before any is used
    RowChunk<T, D, kSmallThreads> cq, ck, cv;
    load_chunk<T, D, kSmallThreads>(cq, Qb, pr.qs[2], r0, pr.N_q, tid);
    if (kv_end > 0) {
      load_chunk<T, D, kSmallThreads>(ck, Kb, pr.ks[2], 0, pr.N_k, tid);
      load_chunk<T, D, kSmallThreads>(cv, Vb, pr.vs[2], 0, pr.N_k, tid);
    }
    store_chunk<T, D, kSmallThreads>(sQ, cq, tid);
    if (kv_end > 0) {
      store_chunk<T, D, kSmallThreads>(sK, ck, tid);
      store_chunk<T, D, kSmallThreads>(sV, cv, tid);
    }
  } else {
    stage_rows_scalar<T, D, kSmallThreads>(sQ, Qb, pr.qs[2], r0, pr.N_q, tid);
  }
  __syncthreads();
  // Q row (scaled) and O accumulator as pairs of columns: the dot products
  // and the P.V updates run on packed fp32x2 FMAs (two FMAs per instruction)
  float2 qr[D / 2];
#pragma unroll
  for (int c = 0; c < D; c += 4) {
    const float4 v = *reinterpret_cast<const float4*>(sQ + qi * LD + c);
    qr[c / 2] = make_float2(v.x * pr.scale_log2, v.y * pr.scale_log2);
    qr[c / 2 + 1] = make_float2(v.z * pr.scale_log2, v.w * pr.scale_log2);
  }
  float2 acc[D / 2];
#pragma unroll
  for (int c = 0; c < D / 2; ++c) acc[c] = make_float2(0.f, 0.f);
  float m = -INFINITY, l = 0.f;
  constexpr int kKeys = 32 / kSmallSplit;  // keys per thread per chunk

#pragma unroll 1
  for (int kc = 0; kc < kv_end; kc += 32) {
    RowChunk<T, D, kSmallThreads> nk, nv;  // the next chunk, loaded while this one is computed
    const bool more = vec && kc + 32 < kv_end;
    if (more) {
      load_chunk<T, D, kSmallThreads>(nk, Kb, pr.ks[2], kc + 32, pr.N_k, tid);
      load_chunk<T, D, kSmallThreads>(nv, Vb, pr.vs[2], kc + 32, pr.N_k, tid);
    }
    if (!vec) {
      __syncthreads();
      stage_rows_scalar<T, D, kSmallThreads>(sK, Kb, pr.ks[2], kc, pr.N_k, tid);
      stage_rows_scalar<T, D, kSmallThreads>(sV, Vb, pr.vs[2], kc, pr.N_k, tid);
      __syncthreads();
    }
    float s[kKeys];
    float mloc = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < kKeys; ++jj) {
      const int kr = jj * kSmallSplit + kt;  // key row of the chunk
      float2 dot2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < D; c += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(sK + kr * LD + c);
        dot2 = ffma2(qr[c / 2], make_float2(k4.x, k4.y), dot2);
        dot2 = ffma2(qr[c / 2 + 1], make_float2(k4.z, k4.w), dot2);
      }
      s[jj] = (kc + kr < vis_end) ? dot2.x + dot2.y : -INFINITY;
      mloc = fmaxf(mloc, s[jj]);
    }
    const float m_new = fmaxf(m, mloc);
    // m = -inf on the first chunk -> 0; a thread that has seen no key keeps 1
    const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
    l *= alpha;
#pragma unroll
    for (int c = 0; c < D / 2; ++c) acc[c] = make_float2(acc[c].x * alpha, acc[c].y * alpha);
#pragma unroll
    for (int jj = 0; jj < kKeys; ++jj) {
      const int kr = jj * kSmallSplit + kt;
      const float p = (kc + kr < vis_end) ? ex2(s[jj] - m_new) : 0.f;
      l += p;
      const float2 p2 = make_float2(p, p);
#pragma unroll
      for (int c = 0; c < D; c += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(sV + kr * LD + c);
        acc[c / 2] = ffma2(p2, make_float2(v4.x, v4.y), acc[c / 2]);
        acc[c / 2 + 1] = ffma2(p2, make_float2(v4.z, v4.w), acc[c / 2 + 1]);
      }
    }
    m = m_new;
    if (more) {
      __syncthreads();
      store_chunk<T, D, kSmallThreads>(sK, nk, tid);
      store_chunk<T, D, kSmallThreads>(sV, nv, tid);
      __syncthreads();
    }
  }

  // merge the row's kSplit partial softmaxes (consecutive lanes of one warp)
  float M = m;
#pragma unroll
  for (int o = 1; o < kSmallSplit; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = (M == -INFINITY || m == -INFINITY) ? 0.f : ex2(m - M);
  l *= w;
#pragma unroll
  for (int o = 1; o < kSmallSplit; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
  for (int c = 0; c < D / 2; ++c) {
    float ax = acc[c].x * w, ay = acc[c].y * w;
#pragma unroll
    for (int o = 1; o < kSmallSplit; o <<= 1) {
      ax += __shfl_xor_sync(0xffffffffu, ax, o);
      ay += __shfl_xor_sync(0xffffffffu, ay, o);
    }
    acc[c] = make_float2(ax, ay);
  }

  // epilogue: O = acc / l through shared memory (each of the row's kSplit
  // threads writes its share of the columns), LSE = (M + log2 l) ln 2
  const float inv = l > 0.f ? 1.f / l : 0.f;  // a row that sees no key: O = 0, LSE = -inf
  __syncthreads();
#pragma unroll
  for (int c = 0; c < D; c += 4)
    if (c / (D / kSmallSplit) == kt)
      *reinterpret_cast<float4*>(sQ + qi * LD + c) =
          make_float4(acc[c / 2].x * inv, acc[c / 2].y * inv, acc[c / 2 + 1].x * inv, acc[c / 2 + 1].y * inv);
  __syncthreads();
  T* Ob = reinterpret_cast<T*>(pr.O) + b * pr.os[0] + h * pr.os[1];
  if (vec) {
    constexpr int V = 16 / sizeof(T);
    constexpr int VPR = D / V;
#pragma unroll
    for (int idx = tid; idx < 32 * VPR; idx += kSmallThreads) {
      const int r = idx / VPR, cv = idx % VPR;
      if (r0 + r >= pr.N_q) continue;
      const float* src = sQ + r * LD + cv * V;
      uint4 wv;
      if constexpr (sizeof(T) == 4) {
        wv = make_uint4(__float_as_uint(src[0]), __float_as_uint(src[1]), __float_as_uint(src[2]),
                        __float_as_uint(src[3]));
      } else {
        wv = make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]),
                        pack_bf16x2(src[4], src[5]), pack_bf16x2(src[6], src[7]));
      }
      *reinterpret_cast<uint4*>(Ob + (long long)(r0 + r) * pr.os[2] + cv * V) = wv;
    }
  } else {
    for (int idx = tid; idx < 32 * D; idx += kSmallThreads) {
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
  if (kt == 0 && q < pr.N_q && pr.LSE)
    pr.LSE[b * pr.ls[0] + h * pr.ls[1] + (long long)q * pr.ls[2]] = (M + __log2f(l)) * 0.69314718055994531f;
}

template <typename T, int D>
constexpr int small_smem_bytes() {
  return 3 * 32 * (D + 4) * static_cast<int>(sizeof(float));
}

}  // namespace fa
