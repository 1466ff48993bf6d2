// fa_bwd.cuh -- FlashAttention-2 backward on the tcgen05 tensor cores (sm_103a).
//
// What it computes ("Blackwell Attention Example", section "Backward Kernel
// Implementation": the row-sum preprocess and the per-tile products of the
// backward kernel; natural-log LSE of the forward here): with
// P = exp(scale * Q K^T - LSE) (rows of the forward's softmax, causal entries
// above the diagonal zero) and the incoming gradient dO,
//     dV = P^T dO,  dP = dO V^T,  delta_i = dO_i . O_i,  dS = P * (dP - delta),
//     dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three launches:
//  * fa_bwd_pre_kernel: delta and LSE * log2(e) per query row into the
//    workspace (padded rows: delta = 0, LSE = +inf, so their P is exactly 0),
//    and the fp32 dQ accumulator zeroed;
//  * fa_bwd_kernel: one work unit = one 128-key tile of one (b, h).  It keeps
//    K_j, V_j in shared memory and dK_j, dV_j in tensor memory, and walks the
//    128-row query tiles that see it: S^T = K_j Q_i^T and dP^T = V_j dO_i^T
//    (lanes = keys), P^T and dS^T by the compute warpgroup, then
//    dV += P^T dO_i and dK += dS^T Q_i with the A operand in tensor memory,
//    and dQ_i = dS K_j with dS^T staged in shared memory (the A operand must
//    have the query rows in lanes, which only the transposed copy provides);
//    dQ_i is added into the fp32 accumulator with vector reductions;
//  * fa_bwd_post_kernel: dQ = scale * accumulator in the output dtype.
//
// Warp roles of fa_bwd_kernel (384 threads): warpgroup 0 = compute (P^T,
// dS^T; thread = key row = tensor-memory lane), warpgroup 1 = epilogue (dQ
// reductions; dK, dV stores at the end of a unit), warp 8 = TMA loads, warp 9
// = MMA issue.  Tensor memory: S^T (then P^T, then dQ) | dP^T (then dS^T) |
// dV | dK.  Every wait is bounded (Watchdog).
#pragma once

#include "fa_ptx.cuh"

namespace fa {

struct BwdParams {
  int B, H, N_q, N_k;
  int causal;
  float scale;            // softmax scale
  float scale_log2;       // scale * log2(e)
  int n_qt, n_kt;         // query / key tiles
  int N_qp;               // N_q rounded up to the query tile
  int n_units;            // B * H * n_kt
  const float* lse2;      // workspace: LSE * log2(e) [B*H][N_qp] (+inf on padding)
  const float* delta;     // workspace: dO . O        [B*H][N_qp] (0 on padding)
  float* dq_acc;          // workspace: fp32 dQ / scale [B*H][N_qp][D]
  void* dK;
  void* dV;
  long long dk_stride[3], dv_stride[3];  // elements: b, h, n
  unsigned int* err;
  unsigned long long timeout_ns;
};

template <int D_>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr int BM = 128;  // query rows per step
  static constexpr int BN = 128;  // keys per work unit (tensor-memory lanes)
  static constexpr int NST = D == 128 ? 1 : 2;  // Q/dO ring depth (shared-memory budget)
  static constexpr int kPanels = D / 64;        // 128-byte swizzle panels of 64 bf16
  static constexpr uint32_t kRowTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr uint32_t kPanelBytes = 128 * 128;      // one panel of a 128-row tile
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kRowTileBytes;
  static constexpr uint32_t kOffQ = kOffV + kRowTileBytes;           // [NST]
  static constexpr uint32_t kOffdO = kOffQ + NST * kRowTileBytes;    // [NST]
  static constexpr uint32_t kOffdS = kOffdO + NST * kRowTileBytes;   // dS^T [keys][queries], 2 panels
  static constexpr uint32_t kOffVec = kOffdS + BN * BM * 2;          // [NST] lse2[BM], delta[BM]
  static constexpr uint32_t kOffBar = kOffVec + NST * 2 * BM * 4;
  static constexpr int kNumBars = 9 + 2 * NST;  // + teardown
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + base alignment slack
  static constexpr uint32_t kThreads = 384;
  // tensor memory columns
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  // instruction descriptors (bf16 inputs, fp32 accumulators)
  static constexpr uint32_t kIdescS = make_idesc(1u, 128, BM, 0, 0);     // K-major A and B
  static constexpr uint32_t kIdescAcc = make_idesc(1u, 128, D, 0, 1);    // A in TMEM, B MN-major
  static constexpr uint32_t kIdescdQ = make_idesc(1u, 128, D, 1, 1);     // A and B MN-major
  static constexpr uint32_t kKVBytes = 2 * kRowTileBytes;
  static constexpr uint32_t kStepBytes = 2 * kRowTileBytes + 2 * BM * 4;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(2 * 128 + 2 * D <= 512, "tensor memory budget");
};

struct BwdBars {
  uint64_t* kv_full;    // [1] K_j, V_j landed
  uint64_t* kv_empty;   // [1] unit's MMAs done with K_j, V_j
  uint64_t* s_full;     // [1] S^T, dP^T ready
  uint64_t* p_full;     // [1] P^T, dS^T written (128 arrivals)
  uint64_t* dq_full;    // [1] dQ_i ready in tensor memory
  uint64_t* dq_empty;   // [1] dQ_i read out (128 arrivals)
  uint64_t* dkv_full;   // [1] unit's dK, dV complete
  uint64_t* dkv_empty;  // [1] dK, dV read out (128 arrivals)
  uint64_t* q_full;     // [NST] Q_i, dO_i, lse2_i, delta_i landed
  uint64_t* q_empty;    // [NST]
};

// Work unit u -> (b*H + h, key tile j).  Causal units are taken in ascending j
// (the longest first: key tile j is seen by query tiles j .. n_qt-1).
struct BwdUnit {
  int bh, b, h, j, i0, n_steps;
};
template <class C>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, int u) {
  BwdUnit w;
  const int BH = p.B * p.H;
  if (p.causal) {
    w.j = u / BH;
    w.bh = u - w.j * BH;
  } else {
    w.bh = u / p.n_kt;
    w.j = u - w.bh * p.n_kt;
  }
  w.b = w.bh / p.H;
  w.h = w.bh - w.b * p.H;
  // first query tile holding a row >= the tile's first key (BM == BN)
  w.i0 = p.causal ? w.j : 0;
  w.n_steps = w.i0 < p.n_qt ? p.n_qt - w.i0 : 0;
  return w;
}

// 1-D bulk copy global -> shared, completing on `bar` (16-byte aligned, size
// a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               ::"l"(dst), "f"(__uint_as_float(a)), "f"(__uint_as_float(b)), "f"(__uint_as_float(c)),
                 "f"(__uint_as_float(d)) : "memory");
}

// ------------------------------------------------------------- pre / post
// One warp per padded query row: delta = dO . O (fp32), lse2 = LSE * log2(e),
// dQ accumulator row zeroed.  Rows past N_q get delta 0 and lse2 +inf.
struct BwdPreParams {
  int B, H, N_q, N_qp;
  const void* O;
  long long o_stride[3];
  const void* dO;
  long long do_stride[3];
  const float* LSE;
  long long lse_stride[3];
  float* lse2;
  float* delta;
  float* dq_acc;
};
template <typename T, int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __grid_constant__ BwdPreParams p) {
  constexpr int PER = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  const long long rows = static_cast<long long>(p.B) * p.H * p.N_qp;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int q = static_cast<int>(row % p.N_qp);
  const long long bh = row / p.N_qp;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  float* acc = p.dq_acc + row * D + lane * PER;
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float dl = 0.f;
  if (q < p.N_q) {
    const T* o = reinterpret_cast<const T*>(p.O) + b * p.o_stride[0] + h * p.o_stride[1] +
                 static_cast<long long>(q) * p.o_stride[2] + lane * PER;
    const T* g = reinterpret_cast<const T*>(p.dO) + b * p.do_stride[0] + h * p.do_stride[1] +
                 static_cast<long long>(q) * p.do_stride[2] + lane * PER;
#pragma unroll
    for (int k = 0; k < PER; ++k) dl = fmaf(static_cast<float>(o[k]), static_cast<float>(g[k]), dl);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, s);
  if (lane == 0) {
    p.delta[row] = dl;
    p.lse2[row] = q < p.N_q ? p.LSE[b * p.lse_stride[0] + h * p.lse_stride[1] +
                                    static_cast<long long>(q) * p.lse_stride[2]] * 1.4426950408889634f
                            : INFINITY;
  }
}

struct BwdPostParams {
  int B, H, N_q, N_qp;
  float scale;
  const float* dq_acc;
  void* dQ;
  long long dq_stride[3];
};
template <typename T, int D>
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const __grid_constant__ BwdPostParams p) {
  constexpr int PER = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  const long long rows = static_cast<long long>(p.B) * p.H * p.N_q;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int q = static_cast<int>(row % p.N_q);
  const long long bh = row / p.N_q;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  const float* src = p.dq_acc + (bh * p.N_qp + q) * D + lane * PER;
  T* dst = reinterpret_cast<T*>(p.dQ) + b * p.dq_stride[0] + h * p.dq_stride[1] +
           static_cast<long long>(q) * p.dq_stride[2] + lane * PER;
#pragma unroll
  for (int k = 0; k < PER; ++k) dst[k] = static_cast<T>(src[k] * p.scale);
}

// ------------------------------------------------------------------ roles
__device__ __forceinline__ bool bwd_warp_wait(uint64_t* bar, uint32_t parity, const Watchdog& wd,
                                              unsigned int where) {
  bool ok = mbar_wait(bar, parity, wd, where);
  return __all_sync(0xffffffffu, ok);
}

template <class C>
__device__ void bwd_load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                              const CUtensorMap* tmdO, const BwdParams& p, uint8_t* smem, const BwdBars& bars,
                              const Watchdog& wd) {
  const uint64_t pol_kv = l2_policy_evict_first();
  const uint64_t pol_q = l2_policy_evict_last();
  uint32_t ku = 0, gs = 0;
  uint32_t kv_armed = 0, q_armed[C::NST] = {};
  bool ok = true;
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    if (w.n_steps == 0) continue;
    if (!(ok = mbar_wait(&bars.kv_empty[0], (ku & 1u) ^ 1u, wd, 0x60))) break;
    mbar_arrive_expect_tx(&bars.kv_full[0], C::kKVBytes);
#pragma unroll
    for (int pn = 0; pn < C::kPanels; ++pn) {
      tma_load_4d(tmK, &bars.kv_full[0], smem + C::kOffK + pn * C::kPanelBytes, pn * 64, w.j * C::BN, w.h, w.b,
                  pol_kv);
      tma_load_4d(tmV, &bars.kv_full[0], smem + C::kOffV + pn * C::kPanelBytes, pn * 64, w.j * C::BN, w.h, w.b,
                  pol_kv);
    }
    ++kv_armed;
    ++ku;
    for (int s = 0; ok && s < w.n_steps; ++s, ++gs) {
      const int i = w.i0 + s;
      const uint32_t st = gs % C::NST;
      if (!(ok = mbar_wait(&bars.q_empty[st], ((gs / C::NST) & 1u) ^ 1u, wd, 0x61))) break;
      mbar_arrive_expect_tx(&bars.q_full[st], C::kStepBytes);
#pragma unroll
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(tmQ, &bars.q_full[st], smem + C::kOffQ + st * C::kRowTileBytes + pn * C::kPanelBytes, pn * 64,
                    i * C::BM, w.h, w.b, pol_q);
        tma_load_4d(tmdO, &bars.q_full[st], smem + C::kOffdO + st * C::kRowTileBytes + pn * C::kPanelBytes,
                    pn * 64, i * C::BM, w.h, w.b, pol_q);
      }
      const long long vrow = static_cast<long long>(w.bh) * p.N_qp + i * C::BM;
      uint8_t* vec = smem + C::kOffVec + st * 2 * C::BM * 4;
      bulk_load(vec, p.lse2 + vrow, C::BM * 4, &bars.q_full[st]);
      bulk_load(vec + C::BM * 4, p.delta + vrow, C::BM * 4, &bars.q_full[st]);
      ++q_armed[st];
    }
  }
  if (!ok) {
    // let copies already in flight land before shared memory goes away
    const uint64_t limit = 100000000ull;
    if (kv_armed) mbar_drain(&bars.kv_full[0], (kv_armed - 1) & 1u, limit);
    for (int st = 0; st < C::NST; ++st)
      if (q_armed[st]) mbar_drain(&bars.q_full[st], (q_armed[st] - 1) & 1u, limit);
  }
}

// K-major operand (a 128-row bf16 tile, K = head dim): k-step kk of 16.
template <class C>
__device__ __forceinline__ uint32_t kmajor_off(int kk) {
  const uint32_t byte = kk * 32;
  return ((byte / 128) * C::kPanelBytes + byte % 128) >> 4;
}

template <class C>
__device__ void bwd_mma_role(const BwdParams& p, uint8_t* smem, uint32_t tmem, const BwdBars& bars,
                             const Watchdog& wd, uint64_t* teardown) {
  const uint32_t k_addr = smem_u32(smem + C::kOffK);
  const uint32_t v_addr = smem_u32(smem + C::kOffV);
  const uint32_t ds_addr = smem_u32(smem + C::kOffdS);
  uint32_t ku = 0, gs = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    if (w.n_steps == 0) continue;
    if (!(ok = bwd_warp_wait(&bars.kv_full[0], ku & 1u, wd, 0x62))) break;
    for (int s = 0; ok && s < w.n_steps; ++s, ++gs) {
      const uint32_t st = gs % C::NST;
      const bool first = (s == 0), last = (s == w.n_steps - 1);
      const uint32_t q_addr = smem_u32(smem + C::kOffQ + st * C::kRowTileBytes);
      const uint32_t do_addr = smem_u32(smem + C::kOffdO + st * C::kRowTileBytes);
      if (!(ok = bwd_warp_wait(&bars.q_full[st], (gs / C::NST) & 1u, wd, 0x63))) break;
      // S^T lands where the previous step's dQ was: wait until it is read out
      if (gs > 0 && !(ok = bwd_warp_wait(&bars.dq_empty[0], (gs - 1) & 1u, wd, 0x64))) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t ak = sdesc_sw128<16, 1024>(k_addr), av = sdesc_sw128<16, 1024>(v_addr);
        const uint64_t bq = sdesc_sw128<16, 1024>(q_addr), bdo = sdesc_sw128<16, 1024>(do_addr);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk)
          mma_ss<false>(tmem + C::kColS, ak + kmajor_off<C>(kk), bq + kmajor_off<C>(kk), C::kIdescS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk)
          mma_ss<false>(tmem + C::kColdP, av + kmajor_off<C>(kk), bdo + kmajor_off<C>(kk), C::kIdescS, kk > 0);
        tc_commit(&bars.s_full[0]);
      }
      __syncwarp();
      if (!(ok = bwd_warp_wait(&bars.p_full[0], gs & 1u, wd, 0x65))) break;
      // the first accumulation of a unit overwrites dK, dV: the previous
      // unit's must have been read out
      if (first && ku > 0 && !(ok = bwd_warp_wait(&bars.dkv_empty[0], (ku - 1) & 1u, wd, 0x66))) break;
      tc_fence_after();
      if (elect_one()) {
        // dV += P^T dO_i, dK += dS^T Q_i: A in tensor memory (bf16 pairs),
        // B MN-major (head dim contiguous, k = query rows in 16-row steps)
        const uint64_t bdo = sdesc_sw128<C::kPanelBytes, 1024>(do_addr);
        const uint64_t bq = sdesc_sw128<C::kPanelBytes, 1024>(q_addr);
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_ts<false>(tmem + C::kColdV, tmem + C::kColS + kk * 8, bdo + ((kk * 16 * 128) >> 4), C::kIdescAcc,
                        (!first || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_ts<false>(tmem + C::kColdK, tmem + C::kColdP + kk * 8, bq + ((kk * 16 * 128) >> 4), C::kIdescAcc,
                        (!first || kk > 0) ? 1u : 0u);
        // dQ_i = dS K_j: A = dS^T in shared memory read MN-major (queries
        // contiguous), B = K_j MN-major (head dim contiguous); k = keys.
        // It overwrites the P^T columns, which the dV MMAs above (issued
        // first, executed in order) have read.
        const uint64_t ads = sdesc_sw128<C::BN * 128, 1024>(ds_addr);
        const uint64_t bk = sdesc_sw128<C::kPanelBytes, 1024>(k_addr);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ss<false>(tmem + C::kColS, ads + ((kk * 16 * 128) >> 4), bk + ((kk * 16 * 128) >> 4), C::kIdescdQ,
                        kk > 0 ? 1u : 0u);
        tc_commit(&bars.dq_full[0]);
        tc_commit(&bars.q_empty[st]);
        if (last) {
          tc_commit(&bars.dkv_full[0]);
          tc_commit(&bars.kv_empty[0]);
        }
      }
      __syncwarp();
    }
    ++ku;
  }
  if (!ok) {
    if (elect_one()) tc_commit(teardown);
    __syncwarp();
    mbar_drain(teardown, 0, 100000000ull);
  }
}

template <class C>
__device__ void bwd_compute_role(const BwdParams& p, uint8_t* smem, uint32_t tmem, const BwdBars& bars,
                                 const Watchdog& wd) {
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int r = wq * 32 + lane;  // key row of the tile = tensor-memory lane
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::kColS;
  const uint32_t tdP = tmem + lane_base + C::kColdP;
  uint8_t* ds_row = smem + C::kOffdS + r * 128;
  const float sc = p.scale_log2;
  const float2 sc2 = make_float2(sc, sc);
  uint32_t gs = 0;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    const int key = w.j * C::BN + r;
    const bool key_ok = key < p.N_k;
    for (int s = 0; s < w.n_steps; ++s, ++gs) {
      const int i = w.i0 + s;
      const uint32_t st = gs % C::NST;
      const float* lse2 = reinterpret_cast<const float*>(smem + C::kOffVec + st * 2 * C::BM * 4);
      const float* dlt = lse2 + C::BM;
      if (!bwd_warp_wait(&bars.s_full[0], gs & 1u, wd, 0x67)) return;
      tc_fence_after();
      // per-element masking only where needed: the key tail, and the
      // diagonal tile of a causal unit (query tails have lse2 = +inf)
      const int q0 = i * C::BM;
      const bool diag = p.causal && q0 < w.j * C::BN + C::BN;
      const bool need_mask = __any_sync(0xffffffffu, !key_ok) || diag;
#pragma unroll 1
      for (int c0 = 0; c0 < C::BM; c0 += 32) {
        uint32_t sv[32], dpv[32];
        tmem_ld32(tS + c0, sv);
        tmem_ld32(tdP + c0, dpv);
        tmem_ld_wait32(sv);
        reg_fence32(dpv);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const int c = c0 + k;
          const float2 l2 = *reinterpret_cast<const float2*>(lse2 + c);
          const float2 dl = *reinterpret_cast<const float2*>(dlt + c);
          const float2 x = ffma2(make_float2(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), sc2,
                                 make_float2(-l2.x, -l2.y));
          float p0 = ex2(x.x), p1 = ex2(x.y);
          if (need_mask) {
            const int q = q0 + c;
            if (!key_ok || (p.causal && key > q)) p0 = 0.f;
            if (!key_ok || (p.causal && key > q + 1)) p1 = 0.f;
          }
          const float ds0 = p0 * (__uint_as_float(dpv[k]) - dl.x);
          const float ds1 = p1 * (__uint_as_float(dpv[k + 1]) - dl.y);
          pw[k / 2] = pack_bf16x2(p0, p1);
          dw[k / 2] = pack_bf16x2(ds0, ds1);
        }
        // P^T and dS^T overwrite S^T and dP^T in place (bf16 pairs: column
        // c/2 < c, whose fp32 values were read above)
        tmem_st16(tS + c0 / 2, pw);
        tmem_st16(tdP + c0 / 2, dw);
        // dS^T row r, queries c0..c0+31, into the 128-byte-swizzled panel
        // layout (64 queries per panel, 8-row groups of 1024 bytes)
        uint8_t* panel = ds_row + (c0 / 64) * (C::BN * 128);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int chunk = ((c0 % 64) / 8 + t) ^ (r & 7);
          *reinterpret_cast<uint4*>(panel + chunk * 16) =
              make_uint4(dw[4 * t], dw[4 * t + 1], dw[4 * t + 2], dw[4 * t + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // dS^T stores -> the tensor core's reads
      tc_fence_before();
      mbar_arrive(&bars.p_full[0]);
    }
  }
}

template <class C>
__device__ void bwd_epilogue_role(const BwdParams& p, uint32_t tmem, const BwdBars& bars, const Watchdog& wd) {
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int r = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  uint32_t ku = 0, gs = 0;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    const int key = w.j * C::BN + r;
    __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(p.dK) + w.b * p.dk_stride[0] +
                            w.h * p.dk_stride[1] + static_cast<long long>(key) * p.dk_stride[2];
    __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(p.dV) + w.b * p.dv_stride[0] +
                            w.h * p.dv_stride[1] + static_cast<long long>(key) * p.dv_stride[2];
    if (w.n_steps == 0) {  // keys no query sees: zero gradients
      if (key < p.N_k)
        for (int c = 0; c < C::D; c += 8) {
          *reinterpret_cast<uint4*>(dk_row + c) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(dv_row + c) = make_uint4(0, 0, 0, 0);
        }
      continue;
    }
    for (int s = 0; s < w.n_steps; ++s, ++gs) {
      const int q = (w.i0 + s) * C::BM + r;
      float* dst = p.dq_acc + (static_cast<long long>(w.bh) * p.N_qp + q) * C::D;
      if (!bwd_warp_wait(&bars.dq_full[0], gs & 1u, wd, 0x68)) return;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < C::D; c += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kColS + c, v);
        tmem_ld_wait32(v);
#pragma unroll
        for (int k = 0; k < 32; k += 4) red_add_v4(dst + c + k, v[k], v[k + 1], v[k + 2], v[k + 3]);
      }
      tc_fence_before();
      mbar_arrive(&bars.dq_empty[0]);
    }
    if (!bwd_warp_wait(&bars.dkv_full[0], ku & 1u, wd, 0x69)) return;
    tc_fence_after();
    const bool valid = key < p.N_k;
#pragma unroll 1
    for (int c = 0; c < C::D; c += 32) {
      uint32_t v[32], k2[32];
      tmem_ld32(tmem + lane_base + C::kColdV + c, v);
      tmem_ld32(tmem + lane_base + C::kColdK + c, k2);
      tmem_ld_wait32(v);
      reg_fence32(k2);
      if (valid) {
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          *reinterpret_cast<uint4*>(dv_row + c + k) =
              make_uint4(pack_bf16x2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])),
                         pack_bf16x2(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])),
                         pack_bf16x2(__uint_as_float(v[k + 4]), __uint_as_float(v[k + 5])),
                         pack_bf16x2(__uint_as_float(v[k + 6]), __uint_as_float(v[k + 7])));
          *reinterpret_cast<uint4*>(dk_row + c + k) =
              make_uint4(pack_bf16x2(__uint_as_float(k2[k]) * p.scale, __uint_as_float(k2[k + 1]) * p.scale),
                         pack_bf16x2(__uint_as_float(k2[k + 2]) * p.scale, __uint_as_float(k2[k + 3]) * p.scale),
                         pack_bf16x2(__uint_as_float(k2[k + 4]) * p.scale, __uint_as_float(k2[k + 5]) * p.scale),
                         pack_bf16x2(__uint_as_float(k2[k + 6]) * p.scale, __uint_as_float(k2[k + 7]) * p.scale));
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&bars.dkv_empty[0]);
    ++ku;
  }
}

template <class C>
__global__ void __launch_bounds__(384, 1)
fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  BwdBars bars;
  bars.kv_full = bar + 0;
  bars.kv_empty = bar + 1;
  bars.s_full = bar + 2;
  bars.p_full = bar + 3;
  bars.dq_full = bar + 4;
  bars.dq_empty = bar + 5;
  bars.dkv_full = bar + 6;
  bars.dkv_empty = bar + 7;
  bars.q_full = bar + 8;
  bars.q_empty = bar + 8 + C::NST;
  uint64_t* teardown = bar + 8 + 2 * C::NST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full[0], 1);
    mbar_init(&bars.kv_empty[0], 1);
    mbar_init(&bars.s_full[0], 1);
    mbar_init(&bars.p_full[0], 128);
    mbar_init(&bars.dq_full[0], 1);
    mbar_init(&bars.dq_empty[0], 128);
    mbar_init(&bars.dkv_full[0], 1);
    mbar_init(&bars.dkv_empty[0], 128);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
    }
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmdO);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{abort_flag, p.err, p.timeout_ns};
  if (warp < 4) {
    bwd_compute_role<C>(p, smem, tmem, bars, wd);
  } else if (warp < 8) {
    bwd_epilogue_role<C>(p, tmem, bars, wd);
  } else if (warp == 8) {
    if (lane == 0) bwd_load_role<C>(&tmQ, &tmK, &tmV, &tmdO, p, smem, bars, wd);
  } else if (warp == 9) {
    bwd_mma_role<C>(p, smem, tmem, bars, wd, teardown);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
