// fa_small_mma.cuh -- the small-head forward (d = 16, 32) for fp32 inputs on
// warp-level tensor-core tiles (mma.sync m16n8k8, tf32 operands, fp32
// accumulators), with fp32 accuracy kept by a three-term split.
//
// Same computation as fa_small.cuh (the online softmax of "Extend Thunder
// with CUDA-Python", flash_attention_reference, base 2 with log2(e) folded
// into the scale as in "Blackwell Attention Example"); same work items, same
// strided, in-place views, same outputs.  Why tensor cores at d = 16: a
// launch of the axial shape moves one memory round trip's worth of data, and
// what follows the loads is a dependent chain of about a thousand fp32 FMAs
// per thread; 16 x 8 x 8 tiles do a 32 x 32 x 16 block product in 16
// instructions.  The tiles are the warp-synchronous kind (no tensor-memory
// set-up): at this size the set-up of the 5th-generation path would cost more
// than the arithmetic.
//
//  * one warp owns 32 query rows of one (problem, b, h); Q, K and V arrive 32
//    rows at a time through shared memory (row pitch D + 4 floats: every
//    fragment load below hits 32 distinct banks), with the loads of the Q
//    block and of the first K/V chunk all in flight before any is used;
//  * fp32 to tf32 without losing accuracy: x = hi + lo with hi = x with its
//    low 13 mantissa bits cleared (a tf32 value) and lo = x - hi (exact), and
//    A B = Ah Bh + Ah Bl + Al Bh up to the Al Bl term (2^-22 relative), so
//    each product is three tile MMAs;
//  * S = Q K^T lands in the accumulator layout (lane (g, t) holds columns 2t
//    and 2t+1 of rows g and g + 8 of each 8-column tile); row max and sum
//    reduce over the lane's columns and the 4 lanes of its quad;
//  * P V takes P straight from those accumulators: the k index of the P.V
//    tile runs over the key columns in the order 0, 2, 4, 6, 1, 3, 5, 7 of
//    each 8-key group, so that the columns a lane holds are the ones its A
//    fragment needs; V's rows are read in the same order (only the shared
//    memory row index changes), so no data moves between lanes;
//  * O accumulates in registers (rescaled by 2^(m_old - m_new) when a chunk
//    raises a row max), leaves through shared memory with coalesced 16-byte
//    stores; LSE (natural log) per row.
#pragma once

#include "fa_small.cuh"

namespace fa {

// x = hi + lo, hi a tf32 value (top 19 bits), lo = x - hi exactly.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  const uint32_t h = __float_as_uint(x) & 0xFFFFE000u;
  hi = h;
  lo = __float_as_uint(x - __uint_as_float(h));
}

// D += A B, one 16 x 8 x 8 tile (A row-major 16 x 8, B 8 x 8 column-major).
__device__ __forceinline__ void mma_16x8x8_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A B in fp32 accuracy from split operands (small terms first).
__device__ __forceinline__ void mma_3xtf32(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                           uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma_16x8x8_tf32(d, al[0], al[1], al[2], al[3], bh0, bh1);
  mma_16x8x8_tf32(d, ah[0], ah[1], ah[2], ah[3], bl0, bl1);
  mma_16x8x8_tf32(d, ah[0], ah[1], ah[2], ah[3], bh0, bh1);
}

template <int D>
constexpr int small_mma_smem_bytes() {
  return 4 * 3 * 32 * (D + 4) * static_cast<int>(sizeof(float));  // 4 warps x (Q, K, V)
}

template <int D>
__global__ void __launch_bounds__(128)
fa_small_mma_kernel(const __grid_constant__ SmallParams P) {
  constexpr int LD = D + 4;
  constexpr int KS = D / 8;  // k-steps of Q K^T = n-tiles of O
  // the next chunk's K/V are loaded into registers during the current chunk
  // at d = 16; at d = 32 they would not fit next to the fragments, so the
  // chunk is loaded when its turn comes
  constexpr bool kPrefetch = D <= 16;
  extern __shared__ float small_mma_smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  float* sQ = small_mma_smem + warp * (3 * 32 * LD);  // Q, later O
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
  const int g = lane >> 2, t = lane & 3;
  const bool vec = pr.vec_ok != 0;

  const float* Qb = reinterpret_cast<const float*>(pr.Q) + b * pr.qs[0] + h * pr.qs[1];
  const int hk = h / pr.kv_group;
  const float* Kb = reinterpret_cast<const float*>(pr.K) + b * pr.ks[0] + hk * pr.ks[1];
  const float* Vb = reinterpret_cast<const float*>(pr.V) + b * pr.vs[0] + hk * pr.vs[1];
  const int kv_end = pr.causal ? min(pr.N_k, r0 + 32 + pr.causal_off) : pr.N_k;  // the warp's keys
  // the four rows of this lane: 16 mi + g + 8 hf
  int vis[2][2];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int q = r0 + 16 * mi + g + 8 * hf;
      vis[mi][hf] = pr.causal ? min(pr.N_k, q + 1 + pr.causal_off) : pr.N_k;  // keys < vis are visible
    }

  if (vec) {
    RowChunk<float, D, 32> cq, ck, cv;
    load_chunk<float, D, 32>(cq, Qb, pr.qs[2], r0, pr.N_q, lane);
    if (kv_end > 0) {
      load_chunk<float, D, 32>(ck, Kb, pr.ks[2], 0, pr.N_k, lane);
      load_chunk<float, D, 32>(cv, Vb, pr.vs[2], 0, pr.N_k, lane);
    }
    store_chunk<float, D, 32>(sQ, cq, lane);
    if (kv_end > 0) {
      store_chunk<float, D, 32>(sK, ck, lane);
      store_chunk<float, D, 32>(sV, cv, lane);
    }
  } else {
    stage_rows_scalar<float, D, 32>(sQ, Qb, pr.qs[2], r0, pr.N_q, lane);
  }
  __syncwarp();

  // Q fragments, split (unscaled: the scale multiplies S)
  uint32_t qh[2][KS][4], ql[2][KS][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const float* r = sQ + (16 * mi + g) * LD + 8 * ks + t;
      split_tf32(r[0], qh[mi][ks][0], ql[mi][ks][0]);
      split_tf32(r[8 * LD], qh[mi][ks][1], ql[mi][ks][1]);
      split_tf32(r[4], qh[mi][ks][2], ql[mi][ks][2]);
      split_tf32(r[8 * LD + 4], qh[mi][ks][3], ql[mi][ks][3]);
    }
  float o[2][KS][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < KS; ++ni)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mi][ni][e] = 0.f;
  float m[2][2], l[2][2];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      m[mi][hf] = -INFINITY;
      l[mi][hf] = 0.f;
    }
  const float sc = pr.scale_log2;

#pragma unroll 1
  for (int kc = 0; kc < kv_end; kc += 32) {
    RowChunk<float, D, 32> nk, nv;  // the next chunk, loaded while this one is computed
    const bool more = kPrefetch && vec && kc + 32 < kv_end;
    if (more) {
      load_chunk<float, D, 32>(nk, Kb, pr.ks[2], kc + 32, pr.N_k, lane);
      load_chunk<float, D, 32>(nv, Vb, pr.vs[2], kc + 32, pr.N_k, lane);
    }
    if (!kPrefetch && vec && kc > 0) {
      __syncwarp();
      load_chunk<float, D, 32>(nk, Kb, pr.ks[2], kc, pr.N_k, lane);
      load_chunk<float, D, 32>(nv, Vb, pr.vs[2], kc, pr.N_k, lane);
      store_chunk<float, D, 32>(sK, nk, lane);
      store_chunk<float, D, 32>(sV, nv, lane);
      __syncwarp();
    }
    if (!vec) {
      __syncwarp();
      stage_rows_scalar<float, D, 32>(sK, Kb, pr.ks[2], kc, pr.N_k, lane);
      stage_rows_scalar<float, D, 32>(sV, Vb, pr.vs[2], kc, pr.N_k, lane);
      __syncwarp();
    }
    // S = Q K^T: 2 row tiles x 4 key tiles of 16 x 8
    float s[2][4][4];
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[mi][ni][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const float* r = sK + (8 * ni + g) * LD + 8 * ks + t;  // B[k][n] = K[key n][dim k]
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(r[0], bh0, bl0);
        split_tf32(r[4], bh1, bl1);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) mma_3xtf32(s[mi][ni], qh[mi][ks], ql[mi][ks], bh0, bh1, bl0, bl1);
      }
    }
    // scale, mask, row max over the lane's columns and its quad
    float mx[2][2];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float v = -INFINITY;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = kc + 8 * ni + 2 * t + e;
            float& x = s[mi][ni][2 * hf + e];
            x = key < vis[mi][hf] ? x * sc : -INFINITY;
            v = fmaxf(v, x);
          }
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        mx[mi][hf] = v;
      }
    // online softmax per row; P replaces S in the accumulators
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float m_new = fmaxf(m[mi][hf], mx[mi][hf]);
        // m = -inf on the first chunk -> 0; a row that has seen no key keeps 1
        const float alpha = m_new == -INFINITY ? 1.f : ex2(m[mi][hf] - m_new);
        l[mi][hf] *= alpha;
#pragma unroll
        for (int ni = 0; ni < KS; ++ni) {
          o[mi][ni][2 * hf] *= alpha;
          o[mi][ni][2 * hf + 1] *= alpha;
        }
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float& x = s[mi][ni][2 * hf + e];
            x = x == -INFINITY ? 0.f : ex2(x - m_new);
            l[mi][hf] += x;
          }
        m[mi][hf] = m_new;
      }
    // O += P V: k-step kt covers keys 8 kt .. 8 kt + 7 in the order 0 2 4 6 1 3 5 7,
    // so that A = P needs exactly the accumulator elements the lane holds
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t ph[2][4], pl[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        split_tf32(s[mi][kt][0], ph[mi][0], pl[mi][0]);  // row g,     k = t     (key 2t)
        split_tf32(s[mi][kt][2], ph[mi][1], pl[mi][1]);  // row g + 8, k = t
        split_tf32(s[mi][kt][1], ph[mi][2], pl[mi][2]);  // row g,     k = t + 4 (key 2t + 1)
        split_tf32(s[mi][kt][3], ph[mi][3], pl[mi][3]);  // row g + 8, k = t + 4
      }
#pragma unroll
      for (int ni = 0; ni < KS; ++ni) {
        const float* r = sV + (8 * kt + 2 * t) * LD + 8 * ni + g;  // B[k][n] = V[key(k)][dim n]
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(r[0], bh0, bl0);   // k = t:     key 2t
        split_tf32(r[LD], bh1, bl1);  // k = t + 4: key 2t + 1
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) mma_3xtf32(o[mi][ni], ph[mi], pl[mi], bh0, bh1, bl0, bl1);
      }
    }
    if (more) {
      __syncwarp();
      store_chunk<float, D, 32>(sK, nk, lane);
      store_chunk<float, D, 32>(sV, nv, lane);
      __syncwarp();
    }
  }

  // epilogue: row sums over the quad, O = acc / l through shared memory,
  // LSE = (m + log2 l) ln 2
  __syncwarp();
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float v = l[mi][hf];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      const float inv = v > 0.f ? 1.f / v : 0.f;  // a row that sees no key: O = 0, LSE = -inf
      const int row = 16 * mi + g + 8 * hf;
#pragma unroll
      for (int ni = 0; ni < KS; ++ni)
        *reinterpret_cast<float2*>(sQ + row * LD + 8 * ni + 2 * t) =
            make_float2(o[mi][ni][2 * hf] * inv, o[mi][ni][2 * hf + 1] * inv);
      const int q = r0 + row;
      if (t == 0 && q < pr.N_q && pr.LSE)
        pr.LSE[b * pr.ls[0] + h * pr.ls[1] + (long long)q * pr.ls[2]] = (m[mi][hf] + __log2f(v)) * 0.69314718055994531f;
    }
  __syncwarp();
  float* Ob = reinterpret_cast<float*>(pr.O) + b * pr.os[0] + h * pr.os[1];
  if (vec) {
    constexpr int VPR = D / 4;
#pragma unroll
    for (int idx = lane; idx < 32 * VPR; idx += 32) {
      const int r = idx / VPR, cv = idx % VPR;
      if (r0 + r >= pr.N_q) continue;
      *reinterpret_cast<float4*>(Ob + (long long)(r0 + r) * pr.os[2] + cv * 4) =
          *reinterpret_cast<const float4*>(sQ + r * LD + cv * 4);
    }
  } else {
    for (int idx = lane; idx < 32 * D; idx += 32) {
      const int r = idx / D, c = idx % D;
      if (r0 + r >= pr.N_q) continue;
      Ob[(long long)(r0 + r) * pr.os[2] + c] = sQ[r * LD + c];
    }
  }
}

}  // namespace fa
