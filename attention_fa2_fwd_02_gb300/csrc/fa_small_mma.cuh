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
//  * two warps own 32 query rows of one (problem, b, h), 16 rows each; Q, K
//    and V arrive 32 rows at a time through shared memory shared by the
//    pair (row pitch D + 4 floats: every
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
  return 2 * 3 * 32 * (D + 4) * static_cast<int>(sizeof(float));  // 2 items x (Q, K, V)
}

// A CTA of four warps works on two items; the two warps of an item each take
// 16 of its 32 query rows and share its Q, K and V tiles in shared memory
// (both warps load them, and a named barrier of the pair orders the copies):
// each warp's chain of dependent tile MMAs is half as long as with one warp per
// item, and twice as many warps are resident.
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
  const int pair = warp >> 1, mi = warp & 1;  // this warp's rows: 16 mi .. 16 mi + 15 of the item
  const int ptid = mi * 32 + lane;            // thread of the pair
  float* sQ = small_mma_smem + pair * (3 * 32 * LD);  // Q, later O
  float* sK = sQ + 32 * LD;
  float* sV = sK + 32 * LD;
  auto pair_sync = [&]() {  // the pair's own named barrier (ids 1 and 2; 0 is __syncthreads)
    if (pair == 0)
      named_barrier_sync(1, 64);
    else
      named_barrier_sync(2, 64);
  };

  const long long item = static_cast<long long>(blockIdx.x) * 2 + pair;
  if (item >= P.n_items) return;  // (the whole pair)
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
  // the item's keys (the same for both warps: they pass the same barriers)
  const int kv_end = pr.causal ? min(pr.N_k, r0 + 32 + pr.causal_off) : pr.N_k;
  // the two rows of this lane: 16 mi + g + 8 hf
  int vis[2];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int q = r0 + 16 * mi + g + 8 * hf;
    vis[hf] = pr.causal ? min(pr.N_k, q + 1 + pr.causal_off) : pr.N_k;  // keys < vis are visible
  }

  if (vec) {
    RowChunk<float, D, 64> cq, ck, cv;
    load_chunk<float, D, 64>(cq, Qb, pr.qs[2], r0, pr.N_q, ptid);
    if (kv_end > 0) {
      load_chunk<float, D, 64>(ck, Kb, pr.ks[2], 0, pr.N_k, ptid);
      load_chunk<float, D, 64>(cv, Vb, pr.vs[2], 0, pr.N_k, ptid);
    }
    store_chunk<float, D, 64>(sQ, cq, ptid);
    if (kv_end > 0) {
      store_chunk<float, D, 64>(sK, ck, ptid);
      store_chunk<float, D, 64>(sV, cv, ptid);
    }
  } else {
    stage_rows_scalar<float, D, 64>(sQ, Qb, pr.qs[2], r0, pr.N_q, ptid);
  }
  pair_sync();

  // Q fragments of this warp's 16 rows, split (unscaled: the scale multiplies S)
  uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const float* r = sQ + (16 * mi + g) * LD + 8 * ks + t;
    split_tf32(r[0], qh[ks][0], ql[ks][0]);
    split_tf32(r[8 * LD], qh[ks][1], ql[ks][1]);
    split_tf32(r[4], qh[ks][2], ql[ks][2]);
    split_tf32(r[8 * LD + 4], qh[ks][3], ql[ks][3]);
  }
  float o[KS][4];
#pragma unroll
  for (int ni = 0; ni < KS; ++ni)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[ni][e] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const float sc = pr.scale_log2;

#pragma unroll 1
  for (int kc = 0; kc < kv_end; kc += 32) {
    RowChunk<float, D, 64> nk, nv;  // the next chunk, loaded while this one is computed
    const bool more = kPrefetch && vec && kc + 32 < kv_end;
    if (more) {
      load_chunk<float, D, 64>(nk, Kb, pr.ks[2], kc + 32, pr.N_k, ptid);
      load_chunk<float, D, 64>(nv, Vb, pr.vs[2], kc + 32, pr.N_k, ptid);
    }
    if (!kPrefetch && vec && kc > 0) {
      pair_sync();
      load_chunk<float, D, 64>(nk, Kb, pr.ks[2], kc, pr.N_k, ptid);
      load_chunk<float, D, 64>(nv, Vb, pr.vs[2], kc, pr.N_k, ptid);
      store_chunk<float, D, 64>(sK, nk, ptid);
      store_chunk<float, D, 64>(sV, nv, ptid);
      pair_sync();
    }
    if (!vec) {
      pair_sync();
      stage_rows_scalar<float, D, 64>(sK, Kb, pr.ks[2], kc, pr.N_k, ptid);
      stage_rows_scalar<float, D, 64>(sV, Vb, pr.vs[2], kc, pr.N_k, ptid);
      pair_sync();
    }
    // S = Q K^T: this warp's 16 rows x 4 key tiles of 8
    float s[4][4];
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[ni][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const float* r = sK + (8 * ni + g) * LD + 8 * ks + t;  // B[k][n] = K[key n][dim k]
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(r[0], bh0, bl0);
        split_tf32(r[4], bh1, bl1);
        mma_3xtf32(s[ni], qh[ks], ql[ks], bh0, bh1, bl0, bl1);
      }
    }
    // scale, mask, row max over the lane's columns and its quad
    float mx[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float v = -INFINITY;
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kc + 8 * ni + 2 * t + e;
          float& x = s[ni][2 * hf + e];
          x = key < vis[hf] ? x * sc : -INFINITY;
          v = fmaxf(v, x);
        }
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      mx[hf] = v;
    }
    // online softmax per row; P replaces S in the accumulators
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float m_new = fmaxf(m[hf], mx[hf]);
      // m = -inf on the first chunk -> 0; a row that has seen no key keeps 1
      const float alpha = m_new == -INFINITY ? 1.f : ex2(m[hf] - m_new);
      l[hf] *= alpha;
#pragma unroll
      for (int ni = 0; ni < KS; ++ni) {
        o[ni][2 * hf] *= alpha;
        o[ni][2 * hf + 1] *= alpha;
      }
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& x = s[ni][2 * hf + e];
          x = x == -INFINITY ? 0.f : ex2(x - m_new);
          l[hf] += x;
        }
      m[hf] = m_new;
    }
    // O += P V: k-step kt covers keys 8 kt .. 8 kt + 7 in the order 0 2 4 6 1 3 5 7,
    // so that A = P needs exactly the accumulator elements the lane holds
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t ph[4], pl[4];
      split_tf32(s[kt][0], ph[0], pl[0]);  // row g,     k = t     (key 2t)
      split_tf32(s[kt][2], ph[1], pl[1]);  // row g + 8, k = t
      split_tf32(s[kt][1], ph[2], pl[2]);  // row g,     k = t + 4 (key 2t + 1)
      split_tf32(s[kt][3], ph[3], pl[3]);  // row g + 8, k = t + 4
#pragma unroll
      for (int ni = 0; ni < KS; ++ni) {
        const float* r = sV + (8 * kt + 2 * t) * LD + 8 * ni + g;  // B[k][n] = V[key(k)][dim n]
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(r[0], bh0, bl0);   // k = t:     key 2t
        split_tf32(r[LD], bh1, bl1);  // k = t + 4: key 2t + 1
        mma_3xtf32(o[ni], ph, pl, bh0, bh1, bl0, bl1);
      }
    }
    if (more) {
      pair_sync();  // both warps are done with this chunk
      store_chunk<float, D, 64>(sK, nk, ptid);
      store_chunk<float, D, 64>(sV, nv, ptid);
      pair_sync();
    }
  }

  // epilogue: row sums over the quad, O = acc / l into this warp's own 16
  // rows of sQ (its Q fragments are in registers), LSE = (m + log2 l) ln 2
  __syncwarp();
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    float v = l[hf];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    const float inv = v > 0.f ? 1.f / v : 0.f;  // a row that sees no key: O = 0, LSE = -inf
    const int row = 16 * mi + g + 8 * hf;
#pragma unroll
    for (int ni = 0; ni < KS; ++ni)
      *reinterpret_cast<float2*>(sQ + row * LD + 8 * ni + 2 * t) =
          make_float2(o[ni][2 * hf] * inv, o[ni][2 * hf + 1] * inv);
    const int q = r0 + row;
    if (t == 0 && q < pr.N_q && pr.LSE)
      pr.LSE[b * pr.ls[0] + h * pr.ls[1] + (long long)q * pr.ls[2]] = (m[hf] + __log2f(v)) * 0.69314718055994531f;
  }
  __syncwarp();
  float* Ob = reinterpret_cast<float*>(pr.O) + b * pr.os[0] + h * pr.os[1];
  if (vec) {
    constexpr int VPR = D / 4;
#pragma unroll
    for (int idx = lane; idx < 16 * VPR; idx += 32) {
      const int r = 16 * mi + idx / VPR, cv = idx % VPR;
      if (r0 + r >= pr.N_q) continue;
      *reinterpret_cast<float4*>(Ob + (long long)(r0 + r) * pr.os[2] + cv * 4) =
          *reinterpret_cast<const float4*>(sQ + r * LD + cv * 4);
    }
  } else {
    for (int idx = lane; idx < 16 * D; idx += 32) {
      const int r = 16 * mi + idx / D, c = idx % D;
      if (r0 + r >= pr.N_q) continue;
      Ob[(long long)(r0 + r) * pr.os[2] + c] = sQ[r * LD + c];
    }
  }
}

}  // namespace fa
