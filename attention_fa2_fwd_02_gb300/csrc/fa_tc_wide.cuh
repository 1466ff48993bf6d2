// fa_tc_wide.cuh -- the FlashAttention-2 forward for head dims above 128 (up
// to 256; bf16), on the 5th-generation tensor cores.
//
// Same computation as fa_tc.cuh (the online softmax of "Extend Thunder with
// CUDA-Python", flash_attention_reference, in the base-2 form of "Blackwell
// Attention Example"), with V and O of up to 256 columns ("Blackwell
// Attention Example", blackwell_attention: Q and K share d, V and O have Dv).
//
// Why a kernel of its own: a 128-row O accumulator of 256 fp32 columns takes
// half of the 512 tensor-memory columns, so the two-stage ping-pong of
// fa_tc.cuh (two query halves, each with its own S and O) no longer fits.
// Here a CTA tile is one 128-row query block, and the overlap comes from
// double-buffered S instead:
//  * tensor memory: S_0 | S_1 (BN columns each) | O (D columns); key tile j
//    uses S_{j mod 2}, P overwrites it in place;
//  * the MMA warp issues S(0), S(1), then per key tile j: O += P(j) V_j and
//    S(j+2) = Q K_{j+2}^T, so the softmax of tile j+1 runs while the tensor
//    core computes P(j) V_j and S(j+2) (tcgen05 MMAs from one thread execute in
//    order: S(j+2) cannot overwrite P(j) before the P.V that reads it);
//  * one softmax warpgroup (thread = query row); a lazy rescale of O (the
//    running max moves only by more than kTau) waits for the P.V in flight to
//    finish before it scales O;
//  * ring order of the K/V tiles: K_0, K_1, then V_j, K_{j+2} -- the order in
//    which the MMA warp consumes them;
//  * warpgroup 1 has no role (its registers go to the softmax);
//  * every wait is bounded (Watchdog), as in fa_tc.cuh.
#pragma once

#include "fa_tc.cuh"

namespace fa {

template <int D_, int BN_, int NSLOT_>
struct TcWideCfg {
  using Elem = __nv_bfloat16;
  static constexpr bool kTF32 = false;
  static constexpr bool kVt = false;
  static constexpr int E = 2;
  static constexpr int D = D_;
  static constexpr int BN = BN_;
  static constexpr int NSLOT = NSLOT_;
  static constexpr int BM = 128;                 // query rows of a CTA tile = TMEM lanes
  static constexpr int kPanelElems = 64;         // bf16 values per 128-byte swizzle row
  static constexpr int kPanels = D / kPanelElems;
  static constexpr int kKStep = 16;              // K extent of one kind::f16 MMA
  static constexpr uint32_t kQPanelBytes = BM * 128;
  static constexpr uint32_t kKVPanelBytes = BN * 128;
  static constexpr uint32_t kVtPanelBytes = 0;
  static constexpr uint32_t kQBytes = BM * D * E;
  static constexpr uint32_t kKVBytes = BN * D * E;
  // tensor-memory columns: S_0 | S_1 | O
  __host__ __device__ static constexpr uint32_t col_s(uint32_t b) { return b * BN; }
  static constexpr uint32_t kColO = 2 * BN;
  static constexpr uint32_t kTmemCols = 512;
  // shared memory: Q, the K/V ring, barriers, row statistics
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = kQBytes;
  static constexpr uint32_t kOffBar = kOffKV + NSLOT * kKVBytes;
  static constexpr int kNumBars = 11 + 2 * NSLOT + 1;
  static constexpr uint32_t kOffStats = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffMisc = kOffStats + BM * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + base alignment slack
  static constexpr uint32_t kIdescS = make_idesc(1u, 128, BN, 0, 0);
  static constexpr uint32_t kIdescO = make_idesc(1u, 128, D, 0, 1);
  static constexpr int kThreads = 512;
  // Register split (setmaxnreg): 128 registers x 512 threads at launch; the
  // four warpgroups' shares add up to 4 x 128.  The softmax raises its share
  // (setmaxnreg.inc), the others lower theirs (setmaxnreg.dec only lowers).
  static constexpr uint32_t kRegSoftmax = 232;
  static constexpr uint32_t kRegIdle = 56;
  static constexpr uint32_t kRegEpilogue = 112;
  static constexpr uint32_t kRegProducer = 112;
  static_assert(kRegSoftmax + kRegIdle + kRegEpilogue + kRegProducer == 4 * 128, "register split");
  static_assert(kRegSoftmax >= 128 && kRegSoftmax <= 256 && kRegSoftmax % 8 == 0, "setmaxnreg.inc share");
  static_assert(kRegIdle <= 128 && kRegEpilogue <= 128 && kRegProducer <= 128, "setmaxnreg.dec shares");
  static_assert(kRegIdle >= 24 && kRegIdle % 8 == 0 && kRegEpilogue % 8 == 0 && kRegProducer % 8 == 0,
                "setmaxnreg share granularity");
  static_assert(D % kPanelElems == 0 && D <= 256, "head dim: whole swizzle rows, at most 256 (MMA N)");
  static_assert(BN % 32 == 0 && BN <= 256, "key tile");
  static_assert(2 * BN + D <= 512, "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct WideBars {
  uint64_t* q_full;    // TMA -> MMA
  uint64_t* q_empty;   // MMA -> TMA (last S of the tile done)
  uint64_t* s_full;    // [2] MMA -> softmax
  uint64_t* p_full;    // [2] softmax -> MMA (128 arrivals)
  uint64_t* pv_done;   // MMA -> softmax: one completion per P.V (lazy rescale)
  uint64_t* o_full;    // MMA -> epilogue (last P.V of the tile done)
  uint64_t* o_empty;   // epilogue -> MMA (128 arrivals)
  uint64_t* st_full;   // softmax -> epilogue (128 arrivals)
  uint64_t* st_empty;  // epilogue -> softmax (128 arrivals)
  uint64_t* kv_full;   // [NSLOT]
  uint64_t* kv_empty;  // [NSLOT]
  uint64_t* teardown;  // [1]
};

// Tile order as in fa_tc.cuh (head groups for K/V reuse in L2, the blocks of a
// group's heads interleaved, the last -- longest under the causal mask --
// first), with 128-row query blocks: n_qblk = ceil(N_q / 128).
template <class C>
__device__ __forceinline__ TileInfo wide_tile_info(const TcParams& p, int u) {
  const int BH = p.B * p.H;
  const int per_group = p.head_group * p.n_qblk;
  const int g = u / per_group;
  const int r = u - g * per_group;
  const int heads = min(p.head_group, BH - g * p.head_group);
  const int qi = r / heads;
  const int bh = g * p.head_group + (r - qi * heads);
  const int qb = p.causal != kNoCausal ? (p.n_qblk - 1 - qi) : qi;
  TileInfo ti;
  ti.b = bh / p.H;
  ti.h = bh - ti.b * p.H;
  ti.hk = ti.h / p.kv_group;
  ti.q0 = qb * C::BM;
  ti.qrow0 = ti.krow0 = 0;
  ti.len_q = ti.len_k = 0;
  ti.coff = kNoCausal;
  ti.split = 0;
  ti.j0 = 0;
  int kv_end = p.N_k;
  if (p.causal != kNoCausal) kv_end = min(kv_end, min(ti.q0 + C::BM, p.N_q) + p.causal);
  const int n_tot = kv_end > 0 ? (kv_end + C::BN - 1) / C::BN : 0;
  ti.n_kv = n_tot > 0 ? n_tot : 1;  // a block that sees no key takes one fully masked key tile
  return ti;
}

// ------------------------------------------------------------- load warp
template <class C>
__device__ void wide_load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                               const TcParams& p, uint8_t* smem, const WideBars& bars, const Watchdog& wd) {
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  uint32_t it = 0, q_armed = 0, tile_k = 0;
  bool ok = true;
  auto load_kv = [&](const CUtensorMap* map, int j, const TileInfo& ti) -> bool {
    const uint32_t slot = it % C::NSLOT;
    if (!mbar_wait(&bars.kv_empty[slot], ((it / C::NSLOT) & 1u) ^ 1u, wd, 0x81)) return false;
    ++it;
    mbar_arrive_expect_tx(&bars.kv_full[slot], C::kKVBytes);
    uint8_t* dst = smem + C::kOffKV + slot * C::kKVBytes;
#pragma unroll
    for (int pn = 0; pn < C::kPanels; ++pn)
      tma_load_4d(map, &bars.kv_full[slot], dst + pn * C::kKVPanelBytes, pn * C::kPanelElems, j * C::BN, ti.hk,
                  ti.b, pol_kv);
    return true;
  };
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++tile_k) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!(ok = mbar_wait(&bars.q_empty[0], (tile_k & 1u) ^ 1u, wd, 0x80))) break;
    mbar_arrive_expect_tx(&bars.q_full[0], C::kQBytes);
#pragma unroll
    for (int pn = 0; pn < C::kPanels; ++pn)
      tma_load_4d(tmQ, &bars.q_full[0], smem + C::kOffQ + pn * C::kQPanelBytes, pn * C::kPanelElems, ti.q0, ti.h,
                  ti.b, pol_q);
    ++q_armed;
    ok = load_kv(tmK, 0, ti) && (ti.n_kv < 2 || load_kv(tmK, 1, ti));
    for (int j = 0; ok && j < ti.n_kv; ++j)
      ok = load_kv(tmV, j, ti) && (j + 2 >= ti.n_kv || load_kv(tmK, j + 2, ti));
  }
  if (!ok) {
    // let copies in flight land before the CTA's shared memory goes away
    const uint64_t limit = 100000000ull;  // 100 ms
    for (uint32_t i = it > C::NSLOT ? it - C::NSLOT : 0; i < it; ++i)
      mbar_drain(&bars.kv_full[i % C::NSLOT], (i / C::NSLOT) & 1u, limit);
    if (q_armed) mbar_drain(&bars.q_full[0], (q_armed - 1) & 1u, limit);
  }
}

// -------------------------------------------------------------- MMA warp
template <class C>
__device__ void wide_mma_role(const TcParams& p, uint8_t* smem, uint32_t tmem, const WideBars& bars,
                              const Watchdog& wd) {
  const uint32_t q_addr = smem_u32(smem + C::kOffQ);
  const uint32_t kv_base = smem_u32(smem + C::kOffKV);
  uint32_t it = 0, tile_k = 0, g = 0;  // g: S tiles issued so far (all tiles of this CTA)
  bool ok = true;
  auto kv_wait = [&](uint32_t i) -> bool {
    return warp_wait(&bars.kv_full[i % C::NSLOT], (i / C::NSLOT) & 1u, wd, 0x82);
  };
  auto slot_addr = [&](uint32_t i) -> uint32_t { return kv_base + (i % C::NSLOT) * C::kKVBytes; };
  // S(g) = Q K^T into S_{g mod 2}.  The buffer is free: S(g-2) was turned into
  // P(g-2), whose P.V was issued before this MMA.
  auto qk = [&](bool last_of_tile) -> bool {
    const uint32_t ik = it++;
    if (!kv_wait(ik)) return false;
    tc_fence_after();
    if (elect_one()) {
      issue_qk<C>(tmem + C::col_s(g & 1u), opaque(q_addr), slot_addr(ik));
      tc_commit(&bars.s_full[g & 1u]);
      tc_commit(&bars.kv_empty[ik % C::NSLOT]);
      if (last_of_tile) tc_commit(&bars.q_empty[0]);
    }
    __syncwarp();
    ++g;
    return true;
  };
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++tile_k) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    const int n = ti.n_kv;
    const uint32_t g0 = g;  // S index of key tile 0 of this tile
    if (!(ok = warp_wait(&bars.q_full[0], tile_k & 1u, wd, 0x83))) break;
    if (!(ok = qk(n == 1))) break;
    if (n > 1 && !(ok = qk(n == 2))) break;
    for (int j = 0; ok && j < n; ++j) {
      const uint32_t gj = g0 + j;
      const uint32_t iv = it++;
      if (!(ok = warp_wait(&bars.p_full[gj & 1u], (gj >> 1) & 1u, wd, 0x84))) break;
      if (j == 0 && !(ok = warp_wait(&bars.o_empty[0], (tile_k & 1u) ^ 1u, wd, 0x85))) break;
      if (!(ok = kv_wait(iv))) break;
      tc_fence_after();
      if (elect_one()) {
        issue_pv<C>(tmem + C::kColO, tmem + C::col_s(gj & 1u), slot_addr(iv), j > 0);
        tc_commit(&bars.kv_empty[iv % C::NSLOT]);
        tc_commit(&bars.pv_done[0]);
        if (j == n - 1) tc_commit(&bars.o_full[0]);
      }
      __syncwarp();
      if (j + 2 < n) ok = qk(j + 2 == n - 1);
    }
  }
  if (!ok) {
    // every MMA already issued must finish before TMEM is released
    if (elect_one()) tc_commit(&bars.teardown[0]);
    __syncwarp();
    mbar_drain(&bars.teardown[0], 0, 100000000ull);
  }
}

// --------------------------------------------------------- softmax warpgroup
template <class C>
__device__ void wide_softmax_role(const TcParams& p, uint32_t tmem, const WideBars& bars, float2* stats,
                                  const Watchdog& wd) {
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tO = tmem + lane_base + C::kColO;
  const float sc = p.scale_log2;
  uint32_t gs = 0, tile_k = 0;  // gs: key tiles processed so far (= S index)

  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++tile_k) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    const int q = ti.q0 + row;
    const int vis_end = p.causal != kNoCausal ? min(p.N_k, q + 1 + p.causal) : p.N_k;  // keys < vis_end are visible
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < ti.n_kv; ++j, ++gs) {
      const uint32_t b = gs & 1u;
      const uint32_t tS = tmem + lane_base + C::col_s(b);
      if (!warp_wait(&bars.s_full[b], (gs >> 1) & 1u, wd, 0x86)) return;
      tc_fence_after();
      uint32_t s[C::BN];
#pragma unroll
      for (int c = 0; c < C::BN; c += 32) tmem_ld32(tS + c, s + c);
      tmem_ld_wait32(s);
#pragma unroll
      for (int c = 32; c < C::BN; c += 32) reg_fence32(s + c);

      const int lim = vis_end - j * C::BN;  // columns c < lim are visible
      const bool need_mask = __any_sync(0xffffffffu, lim < C::BN);
      constexpr int kAcc = 8;
      float acc[kAcc];
      float mx;
      if (sc >= 0.f) {
#pragma unroll
        for (int a = 0; a < kAcc; ++a) acc[a] = -INFINITY;
#pragma unroll
        for (int c = 0; c < C::BN; c += 2)
          acc[(c / 2) % kAcc] = max3f(acc[(c / 2) % kAcc], c < lim ? __uint_as_float(s[c]) : -INFINITY,
                                      c + 1 < lim ? __uint_as_float(s[c + 1]) : -INFINITY);
#pragma unroll
        for (int w = kAcc / 2; w > 0; w /= 2)
#pragma unroll
          for (int a = 0; a < w; ++a) acc[a] = fmaxf(acc[a], acc[a + w]);
        mx = (acc[0] == -INFINITY) ? -INFINITY : acc[0] * sc;
      } else {
#pragma unroll
        for (int a = 0; a < kAcc; ++a) acc[a] = INFINITY;
#pragma unroll
        for (int c = 0; c < C::BN; c += 2)
          acc[(c / 2) % kAcc] = min3f(acc[(c / 2) % kAcc], c < lim ? __uint_as_float(s[c]) : INFINITY,
                                      c + 1 < lim ? __uint_as_float(s[c + 1]) : INFINITY);
#pragma unroll
        for (int w = kAcc / 2; w > 0; w /= 2)
#pragma unroll
          for (int a = 0; a < w; ++a) acc[a] = fminf(acc[a], acc[a + w]);
        mx = (acc[0] == INFINITY) ? -INFINITY : acc[0] * sc;
      }
      // lazy rescale: move the applied max only when it grows by more than kTau
      const float m_new = fmaxf(m_run, mx);
      const bool bump = m_new > m_run + kTau;
      float alpha = 1.f;
      if (bump) {
        alpha = ex2(m_run - m_new);  // 0 on the first tile (m_run = -inf)
        m_run = m_new;
      }
      l_run *= alpha;
      if (j > 0 && __any_sync(0xffffffffu, bump)) {
        // O holds sum_{i<j-1} P_i V_i plus the P(j-1).V still in flight: wait
        // for it (completion number gs - 1 of pv_done; P.V(j) needs P(j), which
        // is not written yet, so pv_done is at most one completion ahead).
        if (!warp_wait(&bars.pv_done[0], (gs - 1) & 1u, wd, 0x87)) return;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < C::D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          tmem_ld_wait32(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tO + c, o);
        }
      }
      const float2 sc2 = make_float2(sc, sc);
      const float2 nm2 = make_float2(-m_run, -m_run);
      float2 sum2[kAcc / 2];
#pragma unroll
      for (int a = 0; a < kAcc / 2; ++a) sum2[a] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c0 = 0; c0 < C::BN; c0 += 32) {
        float e[32];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const int c = c0 + k;
          const float2 x = ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sc2, nm2);
          float v0 = ex2(x.x), v1 = ex2(x.y);
          if (need_mask) {
            if (c >= lim) v0 = 0.f;
            if (c + 1 >= lim) v1 = 0.f;
          }
          e[k] = v0;
          e[k + 1] = v1;
          sum2[(k / 2) % (kAcc / 2)] = fadd2(sum2[(k / 2) % (kAcc / 2)], make_float2(v0, v1));
        }
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) pw[k] = pack_bf16x2(e[2 * k], e[2 * k + 1]);
        tmem_st16(tS + c0 / 2, pw);
      }
#pragma unroll
      for (int w = kAcc / 4; w > 0; w /= 2)
#pragma unroll
        for (int a = 0; a < w; ++a) sum2[a] = fadd2(sum2[a], sum2[a + w]);
      l_run += sum2[0].x + sum2[0].y;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[b]);
    }
    // row statistics for the epilogue: 1/l and LSE (natural log); l = 0 only
    // for a row that sees no key (then O = 0 and LSE = -inf)
    if (!warp_wait(&bars.st_empty[0], (tile_k & 1u) ^ 1u, wd, 0x88)) return;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    stats[row] = make_float2(inv_l, (m_run + __log2f(l_run)) * kLn2);
    mbar_arrive(&bars.st_full[0]);
  }
}

// ------------------------------------------------------- epilogue warpgroup
template <class C>
__device__ void wide_epilogue_role(const TcParams& p, uint32_t tmem, const WideBars& bars, const float2* stats,
                                   const Watchdog& wd) {
  using T = typename C::Elem;
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const uint32_t tO = tmem + (static_cast<uint32_t>(wq * 32) << 16) + C::kColO;
  uint32_t tile_k = 0;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++tile_k) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!warp_wait(&bars.o_full[0], tile_k & 1u, wd, 0x89)) return;
    if (!warp_wait(&bars.st_full[0], tile_k & 1u, wd, 0x8a)) return;
    tc_fence_after();
    const float2 st = stats[row];
    mbar_arrive(&bars.st_empty[0]);
    const int q = ti.q0 + row;
    const bool valid = q < p.N_q;
    T* orow = reinterpret_cast<T*>(p.O) + ti.b * p.o_stride[0] + ti.h * p.o_stride[1] +
              static_cast<long long>(q) * p.o_stride[2];
    const int dv = p.dv;  // columns of O to store (<= D)
#pragma unroll 1
    for (int c = 0; c < dv; c += 32) {
      uint32_t o[32];
      tmem_ld32(tO + c, o);
      tmem_ld_wait32(o);
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (c + 8 * k >= dv) break;
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * st.x, __uint_as_float(o[8 * k + 1]) * st.x);
          w.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * st.x, __uint_as_float(o[8 * k + 3]) * st.x);
          w.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * st.x, __uint_as_float(o[8 * k + 5]) * st.x);
          w.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * st.x, __uint_as_float(o[8 * k + 7]) * st.x);
          dst[k] = w;
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&bars.o_empty[0]);
    if (valid && p.LSE)
      p.LSE[ti.b * p.lse_stride[0] + ti.h * p.lse_stride[1] + static_cast<long long>(q) * p.lse_stride[2]] = st.y;
  }
}

// ------------------------------------------------------------------ kernel
template <class C>
__global__ void __launch_bounds__(512, 1)
fa_tc_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  WideBars bars;
  bars.q_full = bar + 0;
  bars.q_empty = bar + 1;
  bars.s_full = bar + 2;
  bars.p_full = bar + 4;
  bars.pv_done = bar + 6;
  bars.o_full = bar + 7;
  bars.o_empty = bar + 8;
  bars.st_full = bar + 9;
  bars.st_empty = bar + 10;
  bars.kv_full = bar + 11;
  bars.kv_empty = bar + 11 + C::NSLOT;
  bars.teardown = bar + 11 + 2 * C::NSLOT;
  float2* stats = reinterpret_cast<float2*>(smem + C::kOffStats);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full[0], 1);
    mbar_init(&bars.q_empty[0], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.p_full[b], 128);
    }
    mbar_init(&bars.pv_done[0], 1);
    mbar_init(&bars.o_full[0], 1);
    mbar_init(&bars.o_empty[0], 128);
    mbar_init(&bars.st_full[0], 128);
    mbar_init(&bars.st_empty[0], 128);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(&bars.teardown[0], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{abort_flag, p.err, p.timeout_ns};

  const int wg = warp / 4;
  if (wg == 3) {
    setmaxnreg_dec<C::kRegProducer>();
    if (warp == 12 && lane == 0) wide_load_role<C>(&tmQ, &tmK, &tmV, p, smem, bars, wd);
    if (warp == 13) wide_mma_role<C>(p, smem, tmem, bars, wd);
  } else if (wg == 2) {
    setmaxnreg_dec<C::kRegEpilogue>();
    wide_epilogue_role<C>(p, tmem, bars, stats, wd);
  } else if (wg == 1) {
    setmaxnreg_dec<C::kRegIdle>();
  } else {
    setmaxnreg_inc<C::kRegSoftmax>();
    wide_softmax_role<C>(p, tmem, bars, stats, wd);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
