// fa_tc_wide.cuh -- the FlashAttention-2 forward with one 128-row query
// block per CTA tile, on the 5th-generation tensor cores: bf16 head dims above
// 128 (up to 256), and every fp32 input (kind::tf32, head dims up to 128).
//
// Same computation as fa_tc.cuh (the online softmax of "Extend Thunder with
// CUDA-Python", flash_attention_reference, in the base-2 form of "Blackwell
// Attention Example"), with V and O of up to 256 columns ("Blackwell
// Attention Example", blackwell_attention: Q and K share d, V and O have Dv).
//
// Why a kernel of its own: a 128-row tile of Q, K or V of 512 bytes per row
// (bf16 d = 256, fp32 d = 128) takes 64 KB of shared memory, so two query
// halves (the two-stage ping-pong of fa_tc.cuh) and a K/V ring no longer fit
// next to each other, and at bf16 d = 256 neither do their accumulators in
// tensor memory.  Here a CTA tile is one 128-row query block, and the overlap
// comes from double-buffered S instead:
//  * tensor memory: S_0 | S_1 (BN columns each) | O_0 [| O_1] (D columns; a
//    second O buffer where it fits, so that the first P.V of the next tile
//    need not wait for the epilogue); key tile j uses S_{j mod 2}, P
//    overwrites it in place (bf16 pairs, or tf32-rounded fp32);
//  * the MMA warp issues S(0), S(1), then per key tile j: O += P(j) V_j and
//    S(j+2) = Q K_{j+2}^T, so the softmax of tile j+1 runs while the tensor
//    core computes P(j) V_j and S(j+2) (tcgen05 MMAs from one thread execute in
//    order: S(j+2) cannot overwrite P(j) before the P.V that reads it);
//  * one softmax warpgroup (thread = query row); a lazy rescale of O (the
//    running max moves only by more than kTau) waits for the P.V in flight to
//    finish before it scales O;
//  * ring order of the K/V tiles: K_0, K_1, then V_j, K_{j+2} -- the order in
//    which the MMA warp consumes them;
//  * fp32 inputs: tf32-typed tensor maps round Q, K and V to tf32 during the
//    copy.  The tensor core takes tf32 operands K-major only, so V (keys x
//    dims, dims contiguous) must become V^T (dims x keys, keys contiguous).
//    Two ways:
//    - VT (fa_vt_kernel has written V^T to global memory, once per call):
//      the load warp copies V^T tiles like K tiles (BN / 32 panels of 32
//      keys, each D rows of 128 bytes) and the kernel is the bf16 one with
//      tf32 arithmetic -- Q in shared memory, two O buffers;
//    - otherwise warpgroup 1 transposes each V tile in shared memory -- in
//      its ring slot when the tile is square (D = BN), else into a buffer of
//      its own -- with a lane mapping under which no two lanes of a
//      quarter-warp touch the same bank group (transpose_v_tile), and Q
//      lives in tensor memory, as the A operand of a TS-form Q.K^T, so that
//      the tensor core reads only K from shared memory (the transposer
//      already takes much of the shared-memory bandwidth).  Q's TMA copy
//      goes through the K/V ring like a K tile, and the epilogue warpgroup
//      moves it into tensor memory (row per thread), once the previous
//      tile's last Q.K^T is done; the slot it frees deepens the ring to three
//      tiles of 64 KB.
//    For bf16, V is used in place as an MN-major operand and warpgroup 1 has
//    no role;
//  * the epilogue writes O with TMA stores: each of its warps converts one
//    128-byte column chunk of its 32 rows into a swizzled 4 KB shared-memory
//    buffer (two per warp, so the next chunk is written while the last one's
//    store still reads) and one lane issues the store.  Row-per-thread global
//    stores put 32 rows 512 bytes apart into every store instruction, and
//    their load on the memory pipeline slowed the next tile's softmax;
//  * split-KV instantiations (SPLIT): work unit u is the key range u mod s of
//    tile u / s, and writes a normalised partial O and its LSE to the caller's
//    workspace (merged by fa_combine_kernel), as in fa_tc.cuh;
//  * every wait is bounded (Watchdog), as in fa_tc.cuh.
#pragma once

#include "fa_tc.cuh"

namespace fa {

template <typename T, int D_, int BN_, int NSLOT_, bool SPLIT_ = false, bool VT_ = false>
struct TcWideCfg {
  using Elem = T;
  static constexpr bool kSplit = SPLIT_;
  static constexpr bool kVarlen = false;
  static constexpr bool kTF32 = sizeof(T) == 4;
  static constexpr int E = sizeof(T);
  static constexpr int D = D_;
  static constexpr int BN = BN_;
  static constexpr int NSLOT = NSLOT_;
  static constexpr int BM = 128;                 // query rows of a CTA tile = TMEM lanes
  static constexpr int kPanelElems = 128 / E;    // elements per 128-byte swizzle row
  static constexpr int kPanels = D / kPanelElems;
  static constexpr int kKStep = 32 / E;          // K extent of one MMA (16 bf16, 8 tf32)
  static constexpr uint32_t kQPanelBytes = BM * 128;
  static constexpr uint32_t kKVPanelBytes = BN * 128;
  static constexpr uint32_t kQBytes = BM * D * E;
  static constexpr uint32_t kKVBytes = BN * D * E;
  // fp32: the B operand of P.V is V^T (K-major): panels of 32 keys, each D
  // rows of 128 bytes, copied from global memory (VT) or made by warpgroup 1
  static constexpr bool kVKMajor = kTF32;
  static constexpr bool kVtGlobal = VT_;
  static constexpr bool kTransV = kTF32 && !VT_;
  static constexpr bool kVtInPlace = kTransV && D == BN;
  static constexpr uint32_t kVtPanelBytes = D * 128;
  static constexpr uint32_t kVtBytes = (kTransV && !kVtInPlace) ? D * BN * E : 0;
  // fp32 with the transposer: Q in tensor memory, its tiles delivered through the ring
  static constexpr bool kQTmem = kTransV;
  // tensor-memory columns: S_0 | S_1 | O_0 [| O_1] [| Q]
  static constexpr int kOBufs = kQTmem ? 1 : ((2 * BN + 2 * D <= 512) ? 2 : 1);
  __host__ __device__ static constexpr uint32_t col_s(uint32_t b) { return b * BN; }
  __host__ __device__ static constexpr uint32_t col_o(uint32_t b) { return 2 * BN + b * D; }
  static constexpr uint32_t kColQ = 2 * BN + kOBufs * D;
  static constexpr uint32_t kTmemCols = 512;
  // shared memory: Q (bf16), the K/V ring, V^T (fp32, non-square tiles), barriers, row statistics
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = kQTmem ? 0 : kQBytes;
  static constexpr uint32_t kOffVt = kOffKV + NSLOT * kKVBytes;
  // O leaves through shared memory and TMA stores (unsplit): per epilogue warp
  // two 4 KB buffers, each 32 rows x one 128-byte column chunk
  static constexpr bool kTmaStore = !SPLIT_;
  static constexpr uint32_t kStageBytes = kTmaStore ? 4 * 2 * 32 * 128 : 0;
  static constexpr uint32_t kOffStage = kOffVt + kVtBytes;
  static constexpr uint32_t kOffBar = kOffStage + kStageBytes;
  static constexpr int kNumBars = 15 + 4 * NSLOT + 1;
  static constexpr uint32_t kOffStats = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffMisc = kOffStats + BM * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + base alignment slack
  static constexpr uint32_t kIdescS = make_idesc(kTF32 ? 2u : 1u, 128, BN, 0, 0);
  static constexpr uint32_t kIdescO = make_idesc(kTF32 ? 2u : 1u, 128, D, 0, kVKMajor ? 0u : 1u);
  static constexpr int kThreads = 512;
  // Register split (setmaxnreg): 128 registers x 512 threads at launch; the
  // four warpgroups' shares add up to 4 x 128.  The softmax raises its share
  // (setmaxnreg.inc), the others lower theirs (setmaxnreg.dec only lowers).
  static constexpr uint32_t kRegSoftmax = 232;
  static constexpr uint32_t kRegWg1 = kTransV ? 96 : 56;   // V transposer (fp32) or idle
  static constexpr uint32_t kRegEpilogue = kTransV ? 80 : 112;
  static constexpr uint32_t kRegProducer = kTransV ? 104 : 112;
  static_assert(kRegSoftmax + kRegWg1 + kRegEpilogue + kRegProducer == 4 * 128, "register split");
  static_assert(kRegSoftmax >= 128 && kRegSoftmax <= 256 && kRegSoftmax % 8 == 0, "setmaxnreg.inc share");
  static_assert(kRegWg1 <= 128 && kRegEpilogue <= 128 && kRegProducer <= 128, "setmaxnreg.dec shares");
  static_assert(kRegWg1 >= 24 && kRegWg1 % 8 == 0 && kRegEpilogue % 8 == 0 && kRegProducer % 8 == 0,
                "setmaxnreg share granularity");
  static_assert(D % kPanelElems == 0 && D <= 256, "head dim: whole swizzle rows, at most 256 (MMA N)");
  static_assert(BN % 32 == 0 && BN <= 256, "key tile");
  static_assert(!kTransV || (D % 32 == 0 && BN % 32 == 0), "transpose works on 32 x 32 blocks");
  static_assert(!VT_ || (kTF32 && BN % 32 == 0), "V^T from global memory: fp32, whole 32-key panels");
  static_assert(2 * BN + kOBufs * D + (kQTmem ? D : 0) <= 512, "tensor memory budget");
  static_assert(!kQTmem || (BM == BN && kQBytes == kKVBytes), "Q tiles travel in ring slots");
  static_assert(NSLOT <= 8, "ring slots (the load warp's per-slot bookkeeping)");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct WideBars {
  uint64_t* q_full;    // TMA -> MMA (fp32: -> the epilogue warpgroup, which moves Q to TMEM)
  uint64_t* q_empty;   // MMA -> TMA (last S of the tile done; fp32: -> epilogue, TMEM Q free)
  uint64_t* q_ready;   // fp32: epilogue -> MMA, Q is in tensor memory (128 arrivals)
  uint64_t* s_full;    // [2] MMA -> softmax
  uint64_t* p_full;    // [2] softmax -> MMA (128 arrivals)
  uint64_t* pv_done;   // MMA -> softmax: one completion per P.V (lazy rescale)
  uint64_t* o_full;    // [2] MMA -> epilogue (last P.V of a tile done), per O buffer
  uint64_t* o_empty;   // [2] epilogue -> MMA (128 arrivals), per O buffer
  uint64_t* st_full;   // softmax -> epilogue (128 arrivals)
  uint64_t* st_empty;  // epilogue -> softmax (128 arrivals)
  uint64_t* vt_full;   // [NSLOT] transposer -> MMA: V^T ready (fp32; 128 arrivals); per ring
                       // slot when V^T is made in place, else only [0] (the V^T buffer)
  uint64_t* vt_empty;  // MMA -> transposer: the P.V that read the V^T buffer is done (fp32, not in place)
  uint64_t* kv_full;   // [NSLOT] TMA -> MMA (fp32: V tiles only arrive here, no bytes)
  uint64_t* kv_empty;  // [NSLOT]
  uint64_t* v_full;    // [NSLOT] TMA -> transposer: the bytes of V tiles (fp32)
  uint64_t* teardown;  // [1]
};

// Tile order as in fa_tc.cuh (head groups for K/V reuse in L2, the blocks of a
// group's heads interleaved, the last -- longest under the causal mask --
// first), with 128-row query blocks: n_qblk = ceil(N_q / 128).  Split-KV:
// work unit u is split u % n_split of tile u / n_split; the tile's key tiles
// are cut into min(n_split, #tiles) balanced ranges and the other splits are
// empty (n_kv = 0).
template <class C>
__device__ __forceinline__ TileInfo wide_tile_info(const TcParams& p, int u) {
  if (p.causal != kNoCausal) u = snake_unit(u, p.n_units);
  const int t = C::kSplit ? u / p.n_split : u;
  const int split = C::kSplit ? u - t * p.n_split : 0;
  const int BH = p.B * p.H;
  const int per_group = p.head_group * p.n_qblk;
  const int g = t / per_group;
  const int r = t - g * per_group;
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
  ti.split = split;
  int kv_end = p.N_k;
  if (p.causal != kNoCausal) kv_end = min(kv_end, min(ti.q0 + C::BM, p.N_q) + p.causal);
  const int n_tot = kv_end > 0 ? (kv_end + C::BN - 1) / C::BN : 0;
  if constexpr (!C::kSplit) {
    ti.j0 = 0;
    ti.n_kv = n_tot > 0 ? n_tot : 1;  // a block that sees no key takes one fully masked key tile
    return ti;
  }
  const int s_eff = min(p.n_split, n_tot);
  if (split >= s_eff) {
    ti.j0 = 0;
    ti.n_kv = 0;
  } else {
    ti.j0 = split * n_tot / s_eff;
    ti.n_kv = (split + 1) * n_tot / s_eff - ti.j0;
  }
  return ti;
}

// Work units that take a pipeline phase (split-KV: units with keys).
template <class C>
__device__ __forceinline__ bool wide_counted(const TileInfo& ti) {
  return C::kSplit ? ti.n_kv != 0 : true;
}

// ------------------------------------------------------------- load warp
// fp32 inputs: a V tile's bytes complete on v_full[slot], which only the
// transposer waits on -- every phase of it, in order -- and the load warp
// arrives on kv_full[slot] without bytes, so that the phases of kv_full still
// count every ring entry for the MMA warp's waits on K tiles.  (A waiter that
// skipped phases could see a stale parity and take a K tile for a V tile.)
template <class C>
__device__ void wide_load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                               const TcParams& p, uint8_t* smem, const WideBars& bars, const Watchdog& wd) {
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  uint32_t it = 0, q_armed = 0, tile_k = 0;
  uint32_t withheld = ~0u;   // ring entry skipped by the test hook, if any
  bool vt_ready = false;     // V^T from global memory: the V^T pass has completed
  uint32_t v_loads[C::NSLOT] = {};  // fp32: V tiles issued per slot
  uint32_t last_is_v = 0;    // fp32: bit s = the last entry issued into slot s was a V tile
  uint32_t last_is_q = 0;    // fp32: bit s = ... a Q tile
  bool ok = true;
  auto load_kv = [&](const CUtensorMap* map, int j, const TileInfo& ti, bool withhold, bool is_v) -> bool {
    const uint32_t slot = it % C::NSLOT;
    if (!mbar_wait(&bars.kv_empty[slot], ((it / C::NSLOT) & 1u) ^ 1u, wd, 0x81)) return false;
    ++it;
    if (withhold) {  // test hook: this tile never arrives
      withheld = it - 1;
      return true;
    }
    uint64_t* done = &bars.kv_full[slot];
    if (C::kTransV) {
      last_is_q &= ~(1u << slot);
      if (is_v) {
        done = &bars.v_full[slot];
        ++v_loads[slot];
        last_is_v |= 1u << slot;
      } else {
        last_is_v &= ~(1u << slot);
      }
    }
    mbar_arrive_expect_tx(done, C::kKVBytes);
    uint8_t* dst = smem + C::kOffKV + slot * C::kKVBytes;
    if (C::kVtGlobal && is_v) {
      if (!vt_ready) {  // V^T is written by the kernel ahead of this one on the stream
        griddep_wait();
        vt_ready = true;
      }
      // V^T [B][H_kv][Dv][keys]: BN / 32 panels of 32 keys x D rows (rows past
      // Dv and keys past N_k read as zeros)
#pragma unroll
      for (int pn = 0; pn < C::BN / 32; ++pn)
        tma_load_4d(map, done, dst + pn * C::kVtPanelBytes, (ti.j0 + j) * C::BN + pn * 32, 0, ti.hk, ti.b, pol_kv);
    } else {
#pragma unroll
      for (int pn = 0; pn < C::kPanels; ++pn)
        tma_load_4d(map, done, dst + pn * C::kKVPanelBytes, pn * C::kPanelElems, (ti.j0 + j) * C::BN, ti.hk, ti.b,
                    pol_kv);
    }
    if (C::kTransV && is_v) mbar_arrive(&bars.kv_full[slot]);
    return true;
  };
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!wide_counted<C>(ti)) continue;
    // test hook (host-set flag): the second K tile of work unit 0 (the first
    // tile of block 0; the longest tile under a causal mask) is never delivered
    const bool inject = (p.debug_flags & 1) && u == 0;
    if constexpr (C::kQTmem) {
      // Q into the next ring slot; its bytes complete on q_full, kv_full[slot] gets a plain arrival
      const uint32_t slot = it % C::NSLOT;
      if (!(ok = mbar_wait(&bars.kv_empty[slot], ((it / C::NSLOT) & 1u) ^ 1u, wd, 0x80))) break;
      ++it;
      last_is_q |= 1u << slot;
      last_is_v &= ~(1u << slot);
      mbar_arrive_expect_tx(&bars.q_full[0], C::kQBytes);
#pragma unroll
      for (int pn = 0; pn < C::kPanels; ++pn)
        tma_load_4d(tmQ, &bars.q_full[0], smem + C::kOffKV + slot * C::kKVBytes + pn * C::kQPanelBytes,
                    pn * C::kPanelElems, ti.q0, ti.h, ti.b, pol_q);
      mbar_arrive(&bars.kv_full[slot]);
    } else {
      if (!(ok = mbar_wait(&bars.q_empty[0], (tile_k & 1u) ^ 1u, wd, 0x80))) break;
      mbar_arrive_expect_tx(&bars.q_full[0], C::kQBytes);
#pragma unroll
      for (int pn = 0; pn < C::kPanels; ++pn)
        tma_load_4d(tmQ, &bars.q_full[0], smem + C::kOffQ + pn * C::kQPanelBytes, pn * C::kPanelElems, ti.q0, ti.h,
                    ti.b, pol_q);
    }
    ++q_armed;
    ++tile_k;
    ok = load_kv(tmK, 0, ti, false, false) && (ti.n_kv < 2 || load_kv(tmK, 1, ti, inject, false));
    for (int j = 0; ok && j < ti.n_kv; ++j)
      ok = load_kv(tmV, j, ti, false, true) && (j + 2 >= ti.n_kv || load_kv(tmK, j + 2, ti, false, false));
  }
  if (!ok) {
    // let copies in flight land before the CTA's shared memory goes away (only
    // the last entry of each slot can still be in flight)
    const uint64_t limit = 100000000ull;  // 100 ms
    for (uint32_t i = it > C::NSLOT ? it - C::NSLOT : 0; i < it; ++i) {
      if (i == withheld) continue;
      const uint32_t slot = i % C::NSLOT;
      if (C::kTransV && ((last_is_v >> slot) & 1u))
        mbar_drain(&bars.v_full[slot], (v_loads[slot] - 1) & 1u, limit);
      else if (!(C::kQTmem && ((last_is_q >> slot) & 1u)))
        mbar_drain(&bars.kv_full[slot], (i / C::NSLOT) & 1u, limit);
    }
    if (q_armed) mbar_drain(&bars.q_full[0], (q_armed - 1) & 1u, limit);
  }
}

// -------------------------------------------------------- V^T (fp32 inputs)
// One V tile [BN keys][D] as TMA wrote it (D / 32 panels of BN rows x 128
// bytes, 128-byte swizzle: the 16-byte chunk c of row k sits at chunk
// position c ^ (k & 7)) becomes the K-major V^T [D][BN] (BN / 32 panels of D
// rows x 128 bytes, same swizzle), at dst; dst == src when kInPlace (BN == D:
// V^T then has exactly V's layout with the roles of keys and dims swapped).
//
// Work is split in 4 x 4 sub-blocks (keys 4a..4a+3, dims 4b..4b+3): a lane
// reads the four 16-byte rows of its sub-block, transposes them in registers
// and writes four 16-byte rows of V^T.  A quarter-warp (8 lanes, one 128-byte
// wavefront of a 16-byte access) takes, in round t of a 32 x 32 block, the
// sub-blocks (a, b) = ((i + t) mod 8, i) for its lanes i: the bank groups it
// reads, b ^ ((4a + r) mod 8), and writes, a ^ ((4b + e) mod 8), are then
// eight distinct values for every r and e, so no access has a bank conflict.
// In place, a lane swaps sub-block (a, b) with (b, a): blocks (A, B) and
// (B, A) of 32 x 32 are done together (A < B), and the diagonal blocks take
// rounds 0 (sub-blocks on the diagonal, transposed alone) to 4 (half the
// lanes), so that every pair is swapped exactly once.  kThreads threads (a
// multiple of 8) share the work.
template <int BN, int D, bool kInPlace, int kThreads>
__device__ __forceinline__ void transpose_v_tile(uint8_t* src, uint8_t* dst, int tid) {
  constexpr int kQuarters = kThreads / 8;
  const int quarter = tid >> 3;
  const int i = tid & 7;
  // the 16-byte piece of key row k that holds dims 4b..4b+3
  auto load4 = [&](int a, int b, float4 (&v)[4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int k = 4 * a + r;
      v[r] = *reinterpret_cast<const float4*>(src + (b >> 3) * (BN * 128) + k * 128 + (((b & 7) ^ (k & 7)) << 4));
    }
  };
  // V^T rows 4b..4b+3 (dims), key chunk a: keys 4a..4a+3
  auto store4 = [&](int a, int b, const float4 (&v)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = 4 * b + e;
      const float4 w = e == 0 ? make_float4(v[0].x, v[1].x, v[2].x, v[3].x)
                     : e == 1 ? make_float4(v[0].y, v[1].y, v[2].y, v[3].y)
                     : e == 2 ? make_float4(v[0].z, v[1].z, v[2].z, v[3].z)
                              : make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
      *reinterpret_cast<float4*>(dst + (a >> 3) * (D * 128) + n * 128 + (((a & 7) ^ (n & 7)) << 4)) = w;
    }
  };
  // two work items in flight per lane (item and item + kQuarters): all their
  // loads are issued before any store, so the shared-memory latency of one
  // item hides behind the other's
  if constexpr (!kInPlace) {
    constexpr int kItems = (BN / 32) * (D / 32) * 8;
    auto decode = [&](int item, int& a, int& b) -> bool {
      if (item >= kItems) return false;
      const int sb = item >> 3, t = item & 7;
      a = 8 * (sb / (D / 32)) + ((i + t) & 7);
      b = 8 * (sb % (D / 32)) + i;
      return true;
    };
#pragma unroll 1
    for (int item = quarter; item < kItems; item += 2 * kQuarters) {
      int a0 = 0, b0 = 0, a1 = 0, b1 = 0;
      const bool k0 = decode(item, a0, b0), k1 = decode(item + kQuarters, a1, b1);
      float4 v0[4], v1[4];
      if (k0) load4(a0, b0, v0);
      if (k1) load4(a1, b1, v1);
      if (k0) store4(a0, b0, v0);
      if (k1) store4(a1, b1, v1);
    }
  } else {
    static_assert(BN == D, "in-place transpose needs a square tile");
    constexpr int P = BN / 32;
    constexpr int kOff = P * (P - 1) / 2 * 8;  // rounds of the off-diagonal block pairs
    constexpr int kItems = kOff + P * 5;
    // 0: no work for this lane, 1: a sub-block on the diagonal (transposed
    // alone), 2: a pair (a, b) <-> (b, a)
    auto decode = [&](int item, int& a, int& b) -> int {
      if (item >= kItems) return 0;
      int A, B, t;
      if (item < kOff) {
        int pr = item >> 3;
        t = item & 7;
        A = 0;
        while (pr >= P - 1 - A) {
          pr -= P - 1 - A;
          ++A;
        }
        B = A + 1 + pr;
      } else {
        A = B = (item - kOff) / 5;
        t = (item - kOff) % 5;
        if (t == 4 && i >= 4) return 0;
      }
      a = 8 * A + ((i + t) & 7);
      b = 8 * B + i;
      return (A == B && t == 0) ? 1 : 2;
    };
#pragma unroll 1
    for (int item = quarter; item < kItems; item += 2 * kQuarters) {
      int a0 = 0, b0 = 0, a1 = 0, b1 = 0;
      const int k0 = decode(item, a0, b0), k1 = decode(item + kQuarters, a1, b1);
      float4 v0[4], w0[4], v1[4], w1[4];
      if (k0) load4(a0, b0, v0);
      if (k0 == 2) load4(b0, a0, w0);
      if (k1) load4(a1, b1, v1);
      if (k1 == 2) load4(b1, a1, w1);
      if (k0) store4(a0, b0, v0);  // (a, b)^T lands where (b, a) was
      if (k0 == 2) store4(b0, a0, w0);
      if (k1) store4(a1, b1, v1);
      if (k1 == 2) store4(b1, a1, w1);
    }
  }
}

// The V^T makers (fp32 inputs): warpgroup 1.  (Six warps -- adding the two
// idle warps of the producer warpgroup -- transpose a tile faster on their
// own, but slow the softmax warps that share their schedulers by more.)
constexpr int kTransThreads = 128;

// The V^T makers: transpose each V tile in the order the load
// warp delivers them -- in its ring slot as soon as it lands (vt_full of that
// slot), or into the V^T buffer once the P.V that read the previous V^T is
// done.  Every thread publishes its own writes (proxy fence, then an arrival
// on vt_full, which counts kTransThreads), so no warp ever waits for another one: a
// warp that gives up on a wait cannot leave the others stuck.
template <class C>
__device__ void wide_transpose_role(const TcParams& p, uint8_t* smem, const WideBars& bars, const Watchdog& wd,
                                    int tid) {
  uint32_t it = 0, vcount = 0;
  uint32_t v_seen[C::NSLOT] = {};  // V tiles taken per slot (phases of v_full[slot])
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!wide_counted<C>(ti)) continue;
    it += (C::kQTmem ? 1 : 0) + (ti.n_kv < 2 ? 1 : 2);  // [Q,] K_0 [, K_1]
    for (int j = 0; j < ti.n_kv; ++j, ++vcount) {
      const uint32_t iv = it++;
      if (j + 2 < ti.n_kv) ++it;  // K_{j+2} follows V_j
      const uint32_t slot = iv % C::NSLOT;
      if (!warp_wait(&bars.v_full[slot], v_seen[slot] & 1u, wd, 0x8b)) return;
      ++v_seen[slot];
      if (!C::kVtInPlace && !warp_wait(&bars.vt_empty[0], (vcount & 1u) ^ 1u, wd, 0x8c)) return;
      uint8_t* src = smem + C::kOffKV + slot * C::kKVBytes;
      uint8_t* dst = C::kVtInPlace ? src : smem + C::kOffVt;
      transpose_v_tile<C::BN, C::D, C::kVtInPlace, kTransThreads>(src, dst, tid);
      fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
      mbar_arrive(&bars.vt_full[C::kVtInPlace ? slot : 0]);
    }
  }
}

// -------------------------------------------------------------- MMA warp
// S = Q K^T with Q in tensor memory (TS form, fp32 inputs): A = Q, K columns
// of 32-bit tf32 from tmem_q (one MMA takes 8 of them); B = the K tile,
// K-major in shared memory as in issue_qk.
template <class C>
__device__ __forceinline__ void issue_qk_ts(uint32_t tmem_s, uint32_t tmem_q, uint32_t k_addr) {
  const uint64_t b0 = sdesc_sw128<16, 1024>(k_addr);
#pragma unroll
  for (int kk = 0; kk < C::D / C::kKStep; ++kk) {
    const uint32_t byte = kk * 32;
    const uint32_t b_off = ((byte / 128) * C::kKVPanelBytes + byte % 128) >> 4;
    mma_ts<C::kTF32>(tmem_s, tmem_q + kk * 8, b0 + b_off, C::kIdescS, kk > 0 ? 1u : 0u);
  }
}

template <class C>
__device__ void wide_mma_role(const TcParams& p, uint8_t* smem, uint32_t tmem, const WideBars& bars,
                              const Watchdog& wd) {
  const uint32_t q_addr = smem_u32(smem + C::kOffQ);  // (bf16: Q in shared memory)
  const uint32_t kv_base = smem_u32(smem + C::kOffKV);
  const uint32_t vt_base = smem_u32(smem + C::kOffVt);
  uint32_t it = 0, tile_k = 0, g = 0;  // g: S tiles issued so far (all tiles of this CTA)
  uint32_t vcount = 0;                 // V tiles consumed so far
  uint32_t vt_seen[C::NSLOT] = {};     // fp32, V^T in place: V^T tiles taken per slot
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
      if constexpr (C::kQTmem)
        issue_qk_ts<C>(tmem + C::col_s(g & 1u), tmem + C::kColQ, slot_addr(ik));
      else
        issue_qk<C>(tmem + C::col_s(g & 1u), opaque(q_addr), slot_addr(ik));
      tc_commit(&bars.s_full[g & 1u]);
      tc_commit(&bars.kv_empty[ik % C::NSLOT]);
      if (last_of_tile) tc_commit(&bars.q_empty[0]);
    }
    __syncwarp();
    ++g;
    return true;
  };
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!wide_counted<C>(ti)) continue;
    const int n = ti.n_kv;
    const uint32_t g0 = g;  // S index of key tile 0 of this tile
    const uint32_t ob = tile_k % C::kOBufs;          // O buffer of this tile
    const uint32_t o_par = (tile_k / C::kOBufs) & 1u;
    if constexpr (C::kQTmem) {
      // Q is in tensor memory: its ring slot (read by the epilogue's copy) is free
      const uint32_t iq = it++;
      if (!(ok = warp_wait(&bars.q_ready[0], tile_k & 1u, wd, 0x83))) break;
      if (elect_one()) mbar_arrive(&bars.kv_empty[iq % C::NSLOT]);
      __syncwarp();
    } else {
      if (!(ok = warp_wait(&bars.q_full[0], tile_k & 1u, wd, 0x83))) break;
    }
    ++tile_k;
    if (!(ok = qk(n == 1))) break;
    if (n > 1 && !(ok = qk(n == 2))) break;
    for (int j = 0; ok && j < n; ++j, ++vcount) {
      const uint32_t gj = g0 + j;
      const uint32_t iv = it++;
      if (!(ok = warp_wait(&bars.p_full[gj & 1u], (gj >> 1) & 1u, wd, 0x84))) break;
      if (j == 0 && !(ok = warp_wait(&bars.o_empty[ob], o_par ^ 1u, wd, 0x85))) break;
      if constexpr (C::kTransV && C::kVtInPlace)
        ok = warp_wait(&bars.vt_full[iv % C::NSLOT], vt_seen[iv % C::NSLOT]++ & 1u, wd, 0x86);
      else if constexpr (C::kTransV)
        ok = warp_wait(&bars.vt_full[0], vcount & 1u, wd, 0x86);
      else
        ok = kv_wait(iv);
      if (!ok) break;
      const uint32_t v_addr = (C::kTransV && !C::kVtInPlace) ? vt_base : slot_addr(iv);
      tc_fence_after();
      if (elect_one()) {
        // the ring slot of V_j: once V^T sits in its own buffer the slot is
        // free now (the transposer's reads are done); else after the P.V
        if (C::kTransV && !C::kVtInPlace) mbar_arrive(&bars.kv_empty[iv % C::NSLOT]);
        issue_pv<C>(tmem + C::col_o(ob), tmem + C::col_s(gj & 1u), v_addr, j > 0);
        if (C::kTransV && !C::kVtInPlace) tc_commit(&bars.vt_empty[0]);
        if (!C::kTransV || C::kVtInPlace) tc_commit(&bars.kv_empty[iv % C::NSLOT]);
        tc_commit(&bars.pv_done[0]);
        if (j == n - 1) tc_commit(&bars.o_full[ob]);
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
  const float sc = p.scale_log2;
  uint32_t gs = 0, tile_k = 0;  // gs: key tiles processed so far (= S index)

  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!wide_counted<C>(ti)) continue;
    const uint32_t tO = tmem + lane_base + C::col_o(tile_k % C::kOBufs);
    const int q = ti.q0 + row;
    const int vis_end = p.causal != kNoCausal ? min(p.N_k, q + 1 + p.causal) : p.N_k;  // keys < vis_end are visible
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < ti.n_kv; ++j, ++gs) {
      const uint32_t b = gs & 1u;
      const uint32_t tS = tmem + lane_base + C::col_s(b);
      if (!warp_wait(&bars.s_full[b], (gs >> 1) & 1u, wd, 0x87)) return;
      tc_fence_after();
      uint32_t s[C::BN];
#pragma unroll
      for (int c = 0; c < C::BN; c += 32) tmem_ld32(tS + c, s + c);
      tmem_ld_wait32(s);
#pragma unroll
      for (int c = 32; c < C::BN; c += 32) reg_fence32(s + c);

      const int lim = vis_end - (ti.j0 + j) * C::BN;  // columns c < lim are visible
      const bool need_mask = __any_sync(0xffffffffu, lim < C::BN);
      constexpr int kAcc = 8;
      float acc[kAcc];
      float mx;
      if (sc >= 0.f) {
#pragma unroll
        for (int a = 0; a < kAcc; ++a) acc[a] = -INFINITY;
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < C::BN; c += 2)
            acc[(c / 2) % kAcc] = max3f(acc[(c / 2) % kAcc], c < lim ? __uint_as_float(s[c]) : -INFINITY,
                                        c + 1 < lim ? __uint_as_float(s[c + 1]) : -INFINITY);
        } else {
#pragma unroll
          for (int c = 0; c < C::BN; c += 2)
            acc[(c / 2) % kAcc] = max3f(acc[(c / 2) % kAcc], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
        }
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
        if (!warp_wait(&bars.pv_done[0], (gs - 1) & 1u, wd, 0x88)) return;
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
      auto exp_tile = [&](auto masked) {
#pragma unroll
        for (int c0 = 0; c0 < C::BN; c0 += 32) {
          float e[32];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const int c = c0 + k;
            const float2 x = ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sc2, nm2);
            float v0 = ex2(x.x), v1 = ex2(x.y);
            if constexpr (decltype(masked)::value) {
              if (c >= lim) v0 = 0.f;
              if (c + 1 >= lim) v1 = 0.f;
            }
            if constexpr (C::kTF32) {
              // P to tf32 by dropping the 13 low mantissa bits (one integer op,
              // instead of a conversion on the special-function pipe, which ex2
              // already keeps busy): l then sums exactly the P that P.V uses, so
              // the common shrink of the weights cancels in O / l
              v0 = __uint_as_float(__float_as_uint(v0) & 0xFFFFE000u);
              v1 = __uint_as_float(__float_as_uint(v1) & 0xFFFFE000u);
            }
            e[k] = v0;
            e[k + 1] = v1;
            sum2[(k / 2) % (kAcc / 2)] = fadd2(sum2[(k / 2) % (kAcc / 2)], make_float2(v0, v1));
          }
          if constexpr (C::kTF32) {
            uint32_t pw[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) pw[k] = __float_as_uint(e[k]);
            tmem_st32(tS + c0, pw);
          } else {
            uint32_t pw[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) pw[k] = pack_bf16x2(e[2 * k], e[2 * k + 1]);
            tmem_st16(tS + c0 / 2, pw);
          }
        }
      };
      if (need_mask)
        exp_tile(BoolC<true>{});
      else
        exp_tile(BoolC<false>{});
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
    // for a row that sees no key of the unit (then O = 0 and LSE = -inf)
    if (!warp_wait(&bars.st_empty[0], (tile_k & 1u) ^ 1u, wd, 0x89)) return;
    ++tile_k;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    stats[row] = make_float2(inv_l, (m_run + __log2f(l_run)) * kLn2);
    mbar_arrive(&bars.st_full[0]);
  }
}

// ------------------------------------------------------- epilogue warpgroup
template <class C>
__device__ void wide_epilogue_role(const CUtensorMap* tmO, const TcParams& p, uint8_t* smem, uint32_t tmem,
                                   const WideBars& bars, const float2* stats, const Watchdog& wd) {
  using T = typename C::Elem;
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  uint8_t* stage = smem + C::kOffStage + wq * (2 * 32 * 128);  // this warp's two store buffers
  uint32_t n_st = 0;                                           // chunks this warp has stored
  // O / l of tile number k (this CTA's k-th unit with keys), and its LSE
  auto store_tile = [&](const TileInfo& ti, uint32_t k) -> bool {
    const uint32_t ob = k % C::kOBufs;
    if (!warp_wait(&bars.o_full[ob], (k / C::kOBufs) & 1u, wd, 0x8a)) return false;
    if (!warp_wait(&bars.st_full[0], k & 1u, wd, 0x8d)) return false;
    tc_fence_after();
    const float2 st = stats[row];
    mbar_arrive(&bars.st_empty[0]);
    const uint32_t tO = tmem + lane_base + C::col_o(ob);
    const int q = ti.q0 + row;
    const bool valid = q < p.N_q;
    T* orow = reinterpret_cast<T*>(p.O) + ti.b * p.o_stride[0] + ti.h * p.o_stride[1] +
              static_cast<long long>(q) * p.o_stride[2];
    // split-KV: this unit's normalised partial O (fp32) and LSE go to the
    // workspace; the combine kernel merges the splits into O and LSE
    const long long wrow = (static_cast<long long>(ti.split) * p.B * p.H + ti.b * p.H + ti.h) * p.N_q + q;
    const int dv = C::kSplit ? C::D : p.dv;  // columns of O to store (<= D)
    if constexpr (C::kTmaStore) {
      // rows ti.q0 + 32 wq .. + 31 (TMA drops rows past N_q and columns past Dv)
      const bool any_row = ti.q0 + wq * 32 < p.N_q;
#pragma unroll 1
      for (int c = 0; c < dv; c += C::kPanelElems) {
        uint32_t w[32];  // this row's 128 bytes of the chunk
        if constexpr (C::kTF32) {
          tmem_ld32(tO + c, w);
          tmem_ld_wait32(w);
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * st.x);
        } else {
          uint32_t o[64];
          tmem_ld32(tO + c, o);
          tmem_ld32(tO + c + 32, o + 32);
          tmem_ld_wait32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * st.x, __uint_as_float(o[2 * i + 1]) * st.x);
        }
        if (!any_row) continue;
        uint8_t* buf = stage + (n_st & 1u) * (32 * 128);
        if (n_st >= 2) {  // the store that last read this buffer
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
        }
        // row `lane` of the buffer, 16-byte chunk i at position i ^ (row mod 8)
        // (the 128-byte swizzle of the tensor map)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<uint4*>(buf + lane * 128 + ((i ^ (lane & 7)) << 4)) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(tmO, buf, c, ti.q0 + wq * 32, ti.h, ti.b);
          bulk_commit();
        }
        ++n_st;
      }
    }
#pragma unroll 1
    for (int c = 0; !C::kTmaStore && c < dv; c += 32) {
      uint32_t o[32];
      tmem_ld32(tO + c, o);
      tmem_ld_wait32(o);
      if (!valid) continue;
      if constexpr (C::kSplit || C::kTF32) {
        float4* dst = C::kSplit ? reinterpret_cast<float4*>(p.ws_o + wrow * C::D + c)
                                : reinterpret_cast<float4*>(reinterpret_cast<float*>(orow) + c);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (c + 4 * k < dv)
            dst[k] = make_float4(__uint_as_float(o[4 * k]) * st.x, __uint_as_float(o[4 * k + 1]) * st.x,
                                 __uint_as_float(o[4 * k + 2]) * st.x, __uint_as_float(o[4 * k + 3]) * st.x);
      } else {
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
    mbar_arrive(&bars.o_empty[ob]);
    if (valid && C::kSplit)
      p.ws_lse[wrow] = st.y;
    else if (valid && p.LSE)
      p.LSE[ti.b * p.lse_stride[0] + ti.h * p.lse_stride[1] + static_cast<long long>(q) * p.lse_stride[2]] = st.y;
    return true;
  };
  uint32_t tile_k = 0, it = 0;
  TileInfo prev{};
  bool have_prev = false;
  auto run = [&]() {
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const TileInfo ti = wide_tile_info<C>(p, u);
    if (!wide_counted<C>(ti)) continue;
    if constexpr (C::kQTmem) {
      // this tile's Q: ring slot -> tensor memory, once its bytes have landed
      // and the previous tile's last Q.K^T no longer reads tensor-memory Q;
      // then the previous tile's output (which completes later)
      const uint32_t slot = it % C::NSLOT;
      it += 1 + 2 * ti.n_kv;  // Q, then n K and n V tiles
      if (!warp_wait(&bars.q_full[0], tile_k & 1u, wd, 0x8e)) return;
      if (!warp_wait(&bars.q_empty[0], (tile_k & 1u) ^ 1u, wd, 0x8f)) return;
      tc_fence_after();
      const uint8_t* qs = smem + C::kOffKV + slot * C::kKVBytes;
      const uint32_t tQ = tmem + lane_base + C::kColQ;
#pragma unroll 1
      for (int pn = 0; pn < C::kPanels; ++pn) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(qs + pn * C::kQPanelBytes + row * 128 + ((c ^ (row & 7)) << 4));
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        tmem_st32(tQ + pn * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.q_ready[0]);
      if (have_prev && !store_tile(prev, tile_k - 1)) return;
      prev = ti;
      have_prev = true;
      ++tile_k;
    } else {
      if (!store_tile(ti, tile_k)) return;
      ++tile_k;
    }
  }
  if (C::kQTmem && have_prev) store_tile(prev, tile_k - 1);
  };
  run();
  // the O stores must have read their buffers (and landed) before the CTA's
  // shared memory goes away, on every exit path
  if constexpr (C::kTmaStore) {
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }
}

// ------------------------------------------------------------------ kernel
template <class C>
__global__ void __launch_bounds__(512, 1)
fa_tc_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ TcParams p) {
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
  bars.o_empty = bar + 9;
  bars.st_full = bar + 11;
  bars.st_empty = bar + 12;
  bars.vt_empty = bar + 13;
  bars.q_ready = bar + 14;
  bars.kv_full = bar + 15;
  bars.kv_empty = bar + 15 + C::NSLOT;
  bars.v_full = bar + 15 + 2 * C::NSLOT;
  bars.vt_full = bar + 15 + 3 * C::NSLOT;
  bars.teardown = bar + 15 + 4 * C::NSLOT;
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
      mbar_init(&bars.o_full[b], 1);
      mbar_init(&bars.o_empty[b], 128);
    }
    mbar_init(&bars.pv_done[0], 1);
    mbar_init(&bars.st_full[0], 128);
    mbar_init(&bars.st_empty[0], 128);
    mbar_init(&bars.vt_empty[0], 1);
    mbar_init(&bars.q_ready[0], 128);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.vt_full[s], kTransThreads);
    }
    mbar_init(&bars.teardown[0], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    if (C::kTmaStore) prefetch_tensormap(&tmO);
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
    wide_epilogue_role<C>(&tmO, p, smem, tmem, bars, stats, wd);
  } else if (wg == 1) {
    setmaxnreg_dec<C::kRegWg1>();
    if constexpr (C::kTransV) wide_transpose_role<C>(p, smem, bars, wd, threadIdx.x - 128);
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
