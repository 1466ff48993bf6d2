// fa_tc.cuh -- FlashAttention-2 forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA) for sm_103a.
//
// What it computes (per (b, h), query row i): the online softmax of
// "Extend Thunder with CUDA-Python" (flash_attention_reference: S = scale Q K^T
// tile by tile, running max m and sum l, O rescaled by exp(m_old - m_new),
// final O / l and L = m + log l) in the base-2 form of "Blackwell Attention
// Example" (section "Attention Kernel Implementation": log2(e) folded into the
// scale, exp2 for P and for the correction factor), with the top-left causal
// mask of the former.
//
// This kernel takes bf16 inputs (tcgen05 kind::f16) with head dims up to 128;
// fp32 inputs and wider heads run on the single-stage kernel of fa_tc_wide.cuh.
//
// Design for GB300 (differs from both pages' kernels):
//  * one CTA per SM, persistent; a CTA tile is 256 query rows of one (b, h),
//    split into two 128-row halves ("stages") whose softmax runs on two
//    warpgroups in ping-pong while the tensor core works on the other half;
//  * warp roles: warpgroups 0/1 = softmax of stage 0/1, warpgroup 2 = epilogue
//    (O / l, output stores, LSE), warp 12 = TMA loads, warp 13 = MMA issue;
//  * Q tiles and a ring of K/V tiles arrive by TMA (128-byte swizzle) and are
//    handed over with mbarriers;
//  * S = Q K^T (both K-major in shared memory) and O += P V (P from tensor
//    memory, V MN-major in shared memory) are tcgen05.mma with fp32
//    accumulators in tensor memory; P overwrites S in place;
//  * lazy rescaling: the running max only moves when a row's max grows by more
//    than kTau (log2 units); the exact result is unchanged (m cancels in O/l
//    and LSE uses the m actually applied), P stays <= 2^kTau;
//  * every wait is bounded (Watchdog): a stuck pipeline ends the launch with
//    an error word instead of a hang.
#pragma once

#include "fa_ptx.cuh"

namespace fa {

constexpr float kTau = 8.0f;              // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.69314718055994531f;
// TcParams::causal value for "no causal mask" (the field is the mask's offset
// otherwise; one int keeps the kernel's parameter block at its size)
constexpr int kNoCausal = 0x7fffffff;
// packed variable-length batches: bottom-right alignment per sequence (its
// offset len_k - len_q differs between sequences)
constexpr int kVarlenBottomRight = 0x7ffffffe;
// Packed batches hand out their work units at run time: each launch owns a
// pair of counters next to the device error word (units taken, CTAs done),
// picked round robin among kSchedSlots, and the load warp passes the units
// it takes to the other roles through a kSchedDepth-deep queue in shared
// memory.  The last CTA to finish zeroes its pair for the next launch.
constexpr int kSchedSlots = 64;
constexpr int kSchedDepth = 4;
constexpr int kSchedConsumers = 13;  // arrivals that free a queue entry: MMA warp, 2 x 4 softmax warps, 4 epilogue warps

struct TcParams {
  int B, H, N_q, N_k;
  int causal;             // kNoCausal: no mask; else key j is visible to row i iff j <= i + causal
                          // (0: top-left alignment, N_k - N_q: bottom-right)
  float scale_log2;       // scale * log2(e)
  int n_qblk;             // ceil(N_q / tile rows): 256 (two-stage kernel), 384 (three stages), 128 (single-stage)
  union {
    int n_tiles;          // B * H * n_qblk (host bookkeeping; no kernel reads it)
    int sched_slot;       // varlen: this launch's scheduler counters, err[1 + 2 slot] and err[2 + 2 slot]
  };
  union {
    int n_split;          // split-KV instantiations: key-range splits per tile
    int dv;               // the others: output columns written (V's head dim, <= D; the
                          // columns of Q, K, V past their extents load as zeros)
  };
  int n_units;            // n_tiles * n_split work units
  union {
    float* ws_o;          // split-KV: partial outputs, fp32 [n_split][B*H*N_q][D]
    const int* cu_q;      // varlen: query offsets of the B packed sequences [B+1]
  };
  union {
    float* ws_lse;        // split-KV: partial LSE (natural log), [n_split][B*H*N_q]
    const int* cu_k;      // varlen: key offsets [B+1]
  };
  int head_group;         // heads per schedule group (K/V L2 locality)
  int kv_group;           // query heads per K/V head (grouped-query attention; 1 = none)
  void* O;
  long long o_stride[3];  // elements: b, h, n
  float* LSE;
  long long lse_stride[3];
  unsigned int* err;
  unsigned long long timeout_ns;
  int debug_flags;
};

template <typename T, int D_, int BN_, int NSLOT_, bool SPLIT_ = false, bool VARLEN_ = false, int NST_ = 2>
struct TcCfg {
  using Elem = T;
  // query stages of 128 rows per CTA tile, one softmax warpgroup each.  With
  // three (d = 64: 3 x (96 S + 64 O) tensor-memory columns), warpgroup 2 is a
  // softmax group too and every softmax group writes its own rows of O.
  static constexpr int NST = NST_;
  static constexpr bool kOwnEpilogue = NST > 2;
  // variable-length instantiation: B packed sequences (offsets cu_q, cu_k;
  // N_q, N_k = the packed totals), tiles over B x H x ceil(max_len_q / 256)
  static constexpr bool kVarlen = VARLEN_;
  // split-KV instantiation: work units are key-range parts of a tile and write
  // partial results to the workspace (a separate kernel, so that the plain
  // path compiles without any of it)
  static constexpr bool kSplit = SPLIT_;
  static constexpr bool kTF32 = sizeof(T) == 4;
  static constexpr int E = sizeof(T);
  static constexpr int D = D_;
  static constexpr int BN = BN_;
  static constexpr int NSLOT = NSLOT_;
  static constexpr int BM = 128;                  // rows per stage = TMEM lanes
  static constexpr int kPanelElems = 128 / E;     // elements per 128-byte swizzle row
  static constexpr int kPanels = D / kPanelElems;
  static constexpr int kKStep = 32 / E;           // K extent of one MMA instruction
  static constexpr uint32_t kQPanelBytes = BM * 128;
  static constexpr uint32_t kKVPanelBytes = BN * 128;
  static constexpr uint32_t kQBytes = BM * D * E;
  static constexpr uint32_t kKVBytes = BN * D * E;
  static constexpr int kTileRows = NST * BM;       // query rows of a CTA tile
  // tensor-memory columns: S_0 .. S_{NST-1} | O_0 .. O_{NST-1}   (P_s overwrites S_s)
  __host__ __device__ static constexpr uint32_t col_s(int s) { return s * BN; }
  __host__ __device__ static constexpr uint32_t col_o(int s) { return NST * BN + s * D; }
  static constexpr uint32_t kTmemCols = 512;
  // V is used in place as an MN-major B operand (bf16 only: fp32 inputs run
  // on the single-stage kernel of fa_tc_wide.cuh, which takes V^T)
  static constexpr bool kVKMajor = false;
  // shared memory
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKV = NST * kQBytes;
  // O leaves through TMA stores from a 4 KB buffer per storing warp (32 rows
  // x 128 bytes, 128-byte swizzle).  Split units write fp32 partials and keep
  // per-row stores; in a packed batch, a warp whose 32 rows run past the end
  // of its sequence stores its rows one by one.  Measured: +1..2 % at d = 128
  // and on three stages, -4 % on the two-stage d = 64 (causal) tiles, which
  // keep the per-row stores.
  static constexpr bool kTmaStore = !SPLIT_ && (D_ == 128 || NST_ == 3);
  static constexpr int kStoreWarps = NST == 2 ? 4 : 4 * NST;
  static constexpr uint32_t kStoreBufBytes = 32 * 128;
  static constexpr uint32_t kOffStage = kOffKV + NSLOT * kKVBytes;
  static constexpr uint32_t kStageBytes = kTmaStore ? kStoreWarps * kStoreBufBytes : 0;
  static constexpr uint32_t kOffBar = kOffStage + kStageBytes;
  static constexpr int kNumBars = 8 * NST + 2 * NSLOT + 1;
  static constexpr uint32_t kOffStats = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffMisc = kOffStats + NST * BM * 8;
  // varlen: the unit queue (kSchedDepth ints, then full and empty barriers)
  static constexpr uint32_t kOffSched = kOffMisc + 16;
  static constexpr uint32_t kSchedBytes = VARLEN_ ? 16 + 2 * kSchedDepth * 8 : 0;
  static constexpr uint32_t kSmemBytes = kOffSched + kSchedBytes + 1024;  // + base alignment slack
  static constexpr uint32_t kIdescS = make_idesc(kTF32 ? 2u : 1u, 128, BN, 0, 0);
  static constexpr uint32_t kIdescO = make_idesc(kTF32 ? 2u : 1u, 128, D, 0, 1);
  static constexpr int kThreads = 512;
  // Register split (setmaxnreg) of the 4 warpgroups; 128 registers x 512
  // threads at launch, so the shares must add up to 4 x 128.
  static constexpr uint32_t kRegSoftmax = NST == 2 ? 184 : 144;
  static constexpr uint32_t kRegEpilogue = NST == 2 ? 64 : 0;   // (three stages: no epilogue group)
  static constexpr uint32_t kRegProducer = 80;  // load warp + MMA warp
  static_assert(NST * kRegSoftmax + kRegEpilogue + kRegProducer == 4 * 128, "register split");
  static_assert(NST == 2 || NST == 3, "two or three query stages");
  static_assert(kRegSoftmax >= 128 && kRegEpilogue <= 128 && kRegProducer <= 128,
                "setmaxnreg.inc raises, setmaxnreg.dec lowers");

  static_assert(!kTF32, "fp32 inputs run on the single-stage kernel (fa_tc_wide.cuh)");
  static_assert(D % kPanelElems == 0, "head dim must fill whole swizzle rows");
  static_assert(BN % 32 == 0 && BN <= 256, "key tile");
  static_assert(NST * (BN + D) <= 512, "tensor memory budget");
  static_assert(!(kVarlen && NST != 2), "packed batches: 256-row virtual tiles");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kOffStage % 1024 == 0, "swizzled store buffers need 1024-byte alignment");
  static_assert(!(kSplit && kVarlen), "split-KV and varlen are separate instantiations");
};

struct Bars {            // [NST]: one per query stage
  uint64_t* q_full;     // [NST] TMA -> MMA
  uint64_t* q_empty;    // [NST] MMA -> TMA
  uint64_t* s_full;     // [NST] MMA -> softmax
  uint64_t* p_full;     // [NST] softmax -> MMA  (one arrival per warp)
  uint64_t* o_full;     // [NST] MMA -> epilogue (last P.V of a tile done)
  uint64_t* o_empty;    // [NST] epilogue -> MMA (one arrival per warp)
  uint64_t* st_full;    // [NST] softmax -> epilogue: row stats written (per warp; two stages)
  uint64_t* st_empty;   // [NST] epilogue -> softmax (per warp; two stages)
  uint64_t* kv_full;    // [NSLOT]
  uint64_t* kv_empty;   // [NSLOT]
  uint64_t* teardown;   // [1]
  // varlen: the unit queue (UnitSource)
  volatile int* sq_unit;  // [kSchedDepth]
  uint64_t* sq_full;      // [kSchedDepth] load warp -> roles (1 arrival)
  uint64_t* sq_empty;     // [kSchedDepth] roles -> load warp (kSchedConsumers arrivals)
};

struct TileInfo {
  int b, h, hk, q0;      // hk: the K/V head of query head h; q0: first query row (of the sequence)
  int qrow0, krow0;      // varlen: packed rows of the sequence's first query and key (0 otherwise)
  int len_q, len_k;      // varlen: the sequence's lengths
  int coff;              // varlen: the sequence's causal offset (kNoCausal: none)
  int split;   // key-range split of this work unit
  int j0;      // first key tile of the unit
  int n_kv;    // key tiles of the unit (0: nothing to do)
};

// Tile order: heads are taken in groups of `head_group`; inside a group the
// query blocks of all its heads are interleaved, last (longest under the
// causal mask) first, so that concurrently running CTAs share K/V in L2 and
// the causal work is handed out longest-first.  Work unit u is split
// u % n_split of tile u / n_split: the tile's key tiles are cut into
// min(n_split, #tiles) balanced ranges; the remaining splits are empty.
// Causal schedules (tiles of unequal length, longest first): the work units
// of one round -- one per CTA of the persistent grid -- are dealt in
// alternating directions.  In round k, CTA c takes unit k*G + c for even k and
// k*G + (r - 1 - c) for odd k (r = units in that round), so a CTA that took one
// of the longest tiles of a round takes one of the shortest of the next.  A
// permutation of [0, n_units); every role applies it to the same u.
__device__ __forceinline__ int snake_unit(int u, int n_units) {
  const int G = gridDim.x;
  const int k = u / G;
  if ((k & 1) == 0) return u;
  const int base = k * G;
  const int r = min(G, n_units - base);
  return base + r - 1 - (u - base);
}

template <class C>
__device__ __forceinline__ TileInfo tile_info(const TcParams& p, int u) {
  constexpr int BN = C::BN;
  // (not for packed batches: their blocks are ordered by sequence, and the
  // alternating rounds measured 5 % slower there)
  if (!C::kVarlen && p.causal != kNoCausal) u = snake_unit(u, p.n_units);
  if constexpr (C::kVarlen) {
    // virtual tiles in the order of the batched tiles: groups of head_group
    // (b, h) pairs (sized on the host so that their K/V stay in L2), inside a
    // group the query-block ranks of its heads interleaved (last blocks first
    // when causal); a block past its sequence's end is empty
    TileInfo ti;
    const int BH = p.B * p.H;
    const int per_group = p.head_group * p.n_qblk;
    const int g = u / per_group;
    const int r = u - g * per_group;
    const int heads = min(p.head_group, BH - g * p.head_group);
    const int qi = r / heads;
    const int bh = g * p.head_group + (r - qi * heads);
    const bool causal = p.causal != kNoCausal;
    ti.b = bh / p.H;
    ti.h = bh - ti.b * p.H;
    ti.hk = ti.h / p.kv_group;
    ti.q0 = (causal ? (p.n_qblk - 1 - qi) : qi) * C::kTileRows;
    ti.qrow0 = p.cu_q[ti.b];
    ti.krow0 = p.cu_k[ti.b];
    ti.len_q = p.cu_q[ti.b + 1] - ti.qrow0;
    ti.len_k = p.cu_k[ti.b + 1] - ti.krow0;
    ti.coff = !causal ? kNoCausal : (p.causal == kVarlenBottomRight ? ti.len_k - ti.len_q : 0);
    ti.split = 0;
    ti.j0 = 0;
    if (ti.q0 >= ti.len_q) {
      ti.n_kv = 0;
      return ti;
    }
    int kv_end = ti.len_k;
    if (causal) kv_end = min(kv_end, min(ti.q0 + C::kTileRows, ti.len_q) + ti.coff);
    const int n_tot = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
    ti.n_kv = n_tot > 0 ? n_tot : 1;  // rows that see no key take one masked tile
    return ti;
  }
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
  ti.q0 = qb * C::kTileRows;
  ti.qrow0 = ti.krow0 = 0;
  ti.split = split;
  int kv_end = p.N_k;
  if (p.causal != kNoCausal) kv_end = min(kv_end, min(ti.q0 + C::kTileRows, p.N_q) + p.causal);
  // (bottom-right alignment with N_q > N_k: a tile may see no key at all)
  const int n_tot = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
  if constexpr (!C::kSplit) {
    // A tile that sees no key (bottom-right causal, N_q > N_k) still takes
    // one fully masked key tile: its rows get l = 0, hence O = 0 and
    // LSE = -inf, and no role needs a skip test.
    ti.j0 = 0;
    ti.n_kv = n_tot > 0 ? n_tot : 1;
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

// All 32 lanes wait; the warp proceeds together or aborts together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const Watchdog& wd,
                                          unsigned int where) {
  bool ok = mbar_wait(bar, parity, wd, where);
  return __all_sync(0xffffffffu, ok);
}

// The CTA's work units.  Batched problems: u = blockIdx.x, then every
// gridDim.x-th unit.  Packed batches: the units the load warp takes from the
// launch's counter, in the order it takes them -- the load warp (kProducer)
// pushes each into the queue, every other role pops them in the same order.
// A unit >= n_units ends the sequence; so does an expired wait (the watchdog
// has recorded it and the other roles' waits then give up too).
template <class C, bool kProducer>
struct UnitSource {
  const TcParams& p;
  const Bars& q;
  const Watchdog& wd;
  uint32_t k = 0;  // units taken so far
  __device__ __forceinline__ int first() {
    if constexpr (!C::kVarlen) return blockIdx.x;
    else return take();
  }
  __device__ __forceinline__ int next(int u) {
    if constexpr (!C::kVarlen) return u + gridDim.x;
    else return take();
  }
  __device__ __forceinline__ int take() {
    const uint32_t e = k % kSchedDepth, par = (k / kSchedDepth) & 1u;
    ++k;
    if constexpr (kProducer) {  // one thread
      if (!mbar_wait(&q.sq_empty[e], par ^ 1u, wd, 0x18)) return p.n_units;
      unsigned int* ctr = p.err + 1 + 2 * p.sched_slot;
      const int u = min(static_cast<int>(atomicAdd(ctr, 1u)), p.n_units);
      q.sq_unit[e] = u;
      mbar_arrive(&q.sq_full[e]);  // (release: the unit is visible to the roles that wait on it)
      return u;
    } else {  // whole warps
      if (!warp_wait(&q.sq_full[e], par, wd, 0x19)) return p.n_units;
      const int u = q.sq_unit[e];
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&q.sq_empty[e]);
      return u;
    }
  }
};

// ------------------------------------------------------------- load warp
template <class C>
__device__ void tc_load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             const TcParams& p, uint8_t* smem, const Bars& bars, const Watchdog& wd) {
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  uint32_t it = 0;          // ring entries handed out so far
  uint32_t withheld = ~0u;  // ring entry skipped by the test hook, if any
  uint32_t q_armed[C::NST] = {};  // Q copies issued per stage
  bool ok = true;
  uint32_t tile_k = 0;

  auto load_q = [&](int stage, const TileInfo& ti) -> bool {
    if (!mbar_wait(&bars.q_empty[stage], (tile_k & 1u) ^ 1u, wd, 0x10 + stage)) return false;
    mbar_arrive_expect_tx(&bars.q_full[stage], C::kQBytes);
    uint8_t* dst = smem + C::kOffQ + stage * C::kQBytes;
#pragma unroll
    for (int pn = 0; pn < C::kPanels; ++pn)
      tma_load_4d(tmQ, &bars.q_full[stage], dst + pn * C::kQPanelBytes, pn * C::kPanelElems,
                  ti.qrow0 + ti.q0 + stage * C::BM, ti.h, C::kVarlen ? 0 : ti.b, pol_q);
    ++q_armed[stage];
    return true;
  };
  auto load_kv = [&](const CUtensorMap* map, int j, const TileInfo& ti, bool withhold) -> bool {
    const uint32_t slot = it % C::NSLOT;
    if (!mbar_wait(&bars.kv_empty[slot], ((it / C::NSLOT) & 1u) ^ 1u, wd, 0x12)) return false;
    ++it;
    if (withhold) {  // test hook: this tile never arrives
      withheld = it - 1;
      return true;
    }
    mbar_arrive_expect_tx(&bars.kv_full[slot], C::kKVBytes);
    uint8_t* dst = smem + C::kOffKV + slot * C::kKVBytes;
#pragma unroll
    for (int pn = 0; pn < C::kPanels; ++pn)
      tma_load_4d(map, &bars.kv_full[slot], dst + pn * C::kKVPanelBytes, pn * C::kPanelElems,
                  ti.krow0 + (ti.j0 + j) * C::BN, ti.hk, C::kVarlen ? 0 : ti.b, pol_kv);
    return true;
  };

  uint32_t counted = 0;  // empty work units (split-KV) take no pipeline phase
  UnitSource<C, true> src{p, bars, wd};
  for (int u = src.first(); ok && u < p.n_units; u = src.next(u), tile_k += counted) {
    const TileInfo ti = tile_info<C>(p, u);
    counted = (C::kSplit || C::kVarlen) ? (ti.n_kv != 0) : 1u;
    if (!counted) continue;
    const bool inject = (p.debug_flags & 1) && u == 0;  // test hook: work unit 0 withholds its second K tile
    // Q_0, K_0 (the first S needs both), the other stages' Q, then V_0
    ok = load_q(0, ti) && load_kv(tmK, 0, ti, false);
#pragma unroll
    for (int st = 1; st < C::NST; ++st) ok = ok && load_q(st, ti);
    ok = ok && load_kv(tmV, 0, ti, false);
    for (int j = 1; ok && j < ti.n_kv; ++j)
      ok = load_kv(tmK, j, ti, inject && j == 1) && load_kv(tmV, j, ti, false);
  }
  if (!ok) {
    // Let copies already in flight land before the CTA's shared memory goes away.
    // Only the last NSLOT ring entries can still be in flight.
    const uint64_t limit = 100000000ull;  // 100 ms
    for (uint32_t i = it > C::NSLOT ? it - C::NSLOT : 0; i < it; ++i)
      if (i != withheld) mbar_drain(&bars.kv_full[i % C::NSLOT], (i / C::NSLOT) & 1u, limit);
#pragma unroll
    for (int st = 0; st < C::NST; ++st)
      if (q_armed[st]) mbar_drain(&bars.q_full[st], (q_armed[st] - 1) & 1u, limit);
  }
}

// -------------------------------------------------------------- MMA warp
// The descriptor of each operand is built once per call; every k-step adds a
// compile-time offset to its start-address field (16-byte units; operands
// live below 256 KB so the 14-bit field never carries).  The loops unroll, the
// instruction descriptors are immediates and the values are warp-uniform, so
// issuing costs a few instructions per MMA.
// Copy of a value the compiler may not hoist or rematerialise: keeps the
// per-k-step descriptors of loop-invariant operands (Q) from being precomputed
// into registers for the whole tile loop.
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
  asm volatile("mov.b32 %0, %0;" : "+r"(x));
  return x;
}

template <class C>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint32_t q_addr, uint32_t k_addr) {
  const uint64_t a0 = sdesc_sw128<16, 1024>(opaque(q_addr));
  const uint64_t b0 = sdesc_sw128<16, 1024>(k_addr);
#pragma unroll
  for (int kk = 0; kk < C::D / C::kKStep; ++kk) {
    constexpr uint32_t kStep = 32;  // bytes of K per MMA
    const uint32_t byte = kk * kStep;
    const uint32_t a_off = ((byte / 128) * C::kQPanelBytes + byte % 128) >> 4;
    const uint32_t b_off = ((byte / 128) * C::kKVPanelBytes + byte % 128) >> 4;
    mma_ss<C::kTF32>(tmem_s, a0 + a_off, b0 + b_off, C::kIdescS, kk > 0 ? 1u : 0u);
  }
}

template <class C>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_addr,
                                         bool accumulate) {
  if constexpr (C::kVKMajor) {
    // tf32: V^T is [D][BN] with keys contiguous, a K-major B operand like K in
    // Q.K^T, in panels of 32 keys (kVtPanelBytes apart); one MMA takes 8 keys
    const uint64_t b0 = sdesc_sw128<16, 1024>(v_addr);
#pragma unroll
    for (int kk = 0; kk < C::BN / C::kKStep; ++kk) {
      const uint32_t byte = kk * 32;
      const uint32_t b_off = ((byte / 128) * C::kVtPanelBytes + byte % 128) >> 4;
      mma_ts<C::kTF32>(tmem_o, tmem_p + kk * 8, b0 + b_off, C::kIdescO, (accumulate || kk > 0) ? 1u : 0u);
    }
  } else {
    // bf16: V is [BN keys][D] with D contiguous, an MN-major B operand: LBO =
    // distance between 128-byte column panels, SBO = between 8-key row
    // groups; one MMA takes 16 keys
    const uint64_t b0 = sdesc_sw128<C::kKVPanelBytes, 1024>(v_addr);
#pragma unroll
    for (int kk = 0; kk < C::BN / C::kKStep; ++kk) {
      const uint32_t b_off = (kk * C::kKStep * 128) >> 4;
      mma_ts<C::kTF32>(tmem_o, tmem_p + kk * 8, b0 + b_off, C::kIdescO, (accumulate || kk > 0) ? 1u : 0u);
    }
  }
}

// Executed by the whole MMA warp: waits are warp-wide, one elected lane (always
// the same one, so its tcgen05.commit covers every MMA) issues.
template <class C>
__device__ void tc_mma_role(const TcParams& p, uint8_t* smem, uint32_t tmem, const Bars& bars,
                            const Watchdog& wd) {
  const uint32_t q_addr0 = smem_u32(smem + C::kOffQ);
  const uint32_t kv_base = smem_u32(smem + C::kOffKV);
  uint32_t it = 0, tile_k = 0;
  uint32_t p_par[C::NST] = {};
  bool ok = true;
  auto kv_wait = [&](uint32_t i) -> bool {
    return warp_wait(&bars.kv_full[i % C::NSLOT], (i / C::NSLOT) & 1u, wd, 0x20);
  };
  auto slot_addr = [&](uint32_t i) -> uint32_t { return kv_base + (i % C::NSLOT) * C::kKVBytes; };

  uint32_t counted = 0;  // empty work units (split-KV) take no pipeline phase
  UnitSource<C, false> src{p, bars, wd};
  for (int u = src.first(); ok && u < p.n_units; u = src.next(u), tile_k += counted) {
    const TileInfo ti = tile_info<C>(p, u);
    counted = (C::kSplit || C::kVarlen) ? (ti.n_kv != 0) : 1u;
    if (!counted) continue;
    const uint32_t par_k = tile_k & 1u;
    const int n = ti.n_kv;
    // S_s(0) = Q_s K_0^T for every stage
#pragma unroll
    for (int s = 0; s < C::NST; ++s) {
      if (!(ok = warp_wait(&bars.q_full[s], par_k, wd, 0x21 + s) && (s > 0 || kv_wait(it)))) break;
      tc_fence_after();
      if (elect_one()) {
        issue_qk<C>(tmem + C::col_s(s), q_addr0 + s * C::kQBytes, slot_addr(it));
        tc_commit(&bars.s_full[s]);
        if (n == 1) tc_commit(&bars.q_empty[s]);
        if (s == C::NST - 1) tc_commit(&bars.kv_empty[it % C::NSLOT]);
      }
      __syncwarp();
    }
    if (!ok) break;
    ++it;
    // steady state: O_s += P_s(j-1) V_{j-1}, then S_s(j) = Q_s K_j^T
    for (int j = 1; ok && j <= n; ++j) {
      const uint32_t iv = it, ik = it + 1;
      const bool last = (j == n);
      if (!(ok = kv_wait(iv) && (last || kv_wait(ik)))) break;
      const uint32_t v_addr = slot_addr(iv);
      const uint32_t k_addr = slot_addr(ik);
#pragma unroll
      for (int s = 0; s < C::NST; ++s) {
        if (!(ok = warp_wait(&bars.p_full[s], p_par[s], wd, 0x24 + s))) break;
        p_par[s] ^= 1u;
        if (j == 1 && !(ok = warp_wait(&bars.o_empty[s], par_k ^ 1u, wd, 0x27 + s))) break;
        tc_fence_after();
        if (elect_one()) {
          issue_pv<C>(tmem + C::col_o(s), tmem + C::col_s(s), v_addr, j > 1);
          if (s == C::NST - 1) tc_commit(&bars.kv_empty[iv % C::NSLOT]);
          if (last) {
            tc_commit(&bars.o_full[s]);
          } else {
            issue_qk<C>(tmem + C::col_s(s), q_addr0 + s * C::kQBytes, k_addr);
            tc_commit(&bars.s_full[s]);
            if (j == n - 1) tc_commit(&bars.q_empty[s]);
            if (s == C::NST - 1) tc_commit(&bars.kv_empty[ik % C::NSLOT]);
          }
        }
        __syncwarp();
      }
      if (!ok) break;
      it += last ? 1 : 2;
    }
  }
  if (!ok) {
    // Make sure every MMA already issued has finished before TMEM is released.
    if (elect_one()) tc_commit(&bars.teardown[0]);
    __syncwarp();
    mbar_drain(&bars.teardown[0], 0, 100000000ull);
  }
}

// ------------------------------------------------------- epilogue
// Rows of stage s of tile ti, row `row` of this thread (TMEM lane): O / l
// (O_s read from tensor memory, st.x = 1/l) and the LSE (st.y), then O_s is
// handed back to the MMA warp (o_empty).
template <class C>
__device__ __forceinline__ void store_stage(const TcParams& p, const TileInfo& ti, int s, float2 st,
                                            uint32_t tmem, uint32_t lane_base, int row, const Bars& bars,
                                            const CUtensorMap* tmO, uint8_t* store_buf) {
  using T = typename C::Elem;
  const int q = ti.q0 + s * C::BM + row;
  // varlen: rows of this sequence only, stored at their packed index (the
  // bound on the packed total also keeps bad offsets from writing out of range)
  const int qo = ti.qrow0 + q;
  const bool valid = C::kVarlen ? (q < ti.len_q && qo < p.N_q && ti.qrow0 >= 0) : q < p.N_q;
  const int ob = C::kVarlen ? 0 : ti.b;
  T* orow = reinterpret_cast<T*>(p.O) + ob * p.o_stride[0] + ti.h * p.o_stride[1] +
            static_cast<long long>(qo) * p.o_stride[2];
  // split-KV: this unit's normalised partial O (fp32) and LSE go to the
  // workspace; the combine kernel merges the splits into O and LSE
  constexpr bool partial = C::kSplit;
  const long long wrow = (static_cast<long long>(ti.split) * p.B * p.H + ti.b * p.H + ti.h) * p.N_q + q;
  const uint32_t tO = tmem + lane_base + C::col_o(s);
  const int dv = C::kSplit ? C::D : p.dv;  // columns of O to store
  // this warp's 32 rows (warp-uniform choices)
  const int r0 = ti.q0 + s * C::BM + (row & ~31);
  const bool rows_one_by_one = !C::kTmaStore || (C::kVarlen && r0 + 32 > ti.len_q && r0 < ti.len_q);
  if (C::kTmaStore && !rows_one_by_one) {
    // 64 columns (one swizzle row) per store; the TMA drops rows past the
    // tensor's end and columns past Dv.  Packed batches: rows r0 .. r0 + 31
    // all belong to the sequence here (or none does), at packed rows
    // qrow0 + r0 ..; a negative offset (bad cu_seqlens) stores nothing
    const int lane = row & 31;
    const bool any_row = C::kVarlen ? (r0 < ti.len_q && ti.qrow0 >= 0) : r0 < p.N_q;
#pragma unroll 1
    for (int c = 0; c < dv; c += 64) {
      if (any_row) {  // the store that last read the buffer
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        tmem_ld32(tO + c + 32 * h, o);
        tmem_ld_wait32(o);
        if (!any_row) continue;
        // 16-byte chunk k of row `lane` at position k ^ (lane mod 8)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(store_buf + lane * 128 + (((4 * h + i) ^ (lane & 7)) << 4)) = make_uint4(
              pack_bf16x2(__uint_as_float(o[8 * i + 0]) * st.x, __uint_as_float(o[8 * i + 1]) * st.x),
              pack_bf16x2(__uint_as_float(o[8 * i + 2]) * st.x, __uint_as_float(o[8 * i + 3]) * st.x),
              pack_bf16x2(__uint_as_float(o[8 * i + 4]) * st.x, __uint_as_float(o[8 * i + 5]) * st.x),
              pack_bf16x2(__uint_as_float(o[8 * i + 6]) * st.x, __uint_as_float(o[8 * i + 7]) * st.x));
      }
      if (!any_row) continue;
      fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine's reads
      __syncwarp();
      if (lane == 0) {
        tma_store_4d(tmO, store_buf, c, ti.qrow0 + r0, ti.h, ob);
        bulk_commit();
      }
    }
  }
#pragma unroll 1
  for (int c = 0; rows_one_by_one && c < dv; c += 32) {
    uint32_t o[32];
    tmem_ld32(tO + c, o);
    tmem_ld_wait32(o);
    if (partial && valid) {
      float4* dst = reinterpret_cast<float4*>(p.ws_o + wrow * C::D + c);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        dst[k] = make_float4(__uint_as_float(o[4 * k]) * st.x, __uint_as_float(o[4 * k + 1]) * st.x,
                             __uint_as_float(o[4 * k + 2]) * st.x, __uint_as_float(o[4 * k + 3]) * st.x);
    } else if (valid) {
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
  mbar_arrive_warp(&bars.o_empty[s]);
  if (partial && valid)
    p.ws_lse[wrow] = st.y;
  else if (valid && p.LSE)
    p.LSE[ob * p.lse_stride[0] + ti.h * p.lse_stride[1] + static_cast<long long>(qo) * p.lse_stride[2]] = st.y;
}

// --------------------------------------------------------- softmax warpgroups
template <class C>
__device__ void tc_softmax_role(const TcParams& p, int stage, uint32_t tmem, const Bars& bars,
                                float2* stats, const Watchdog& wd, const CUtensorMap* tmO, uint8_t* smem) {
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lane_base + C::col_s(stage);
  const uint32_t tO = tmem + lane_base + C::col_o(stage);
  const float sc = p.scale_log2;
  uint32_t s_par = 0, tile_k = 0;

  uint32_t counted = 0;  // empty work units (split-KV) take no pipeline phase
  UnitSource<C, false> src{p, bars, wd};
  for (int u = src.first(); u < p.n_units; u = src.next(u), tile_k += counted) {
    const TileInfo ti = tile_info<C>(p, u);
    counted = (C::kSplit || C::kVarlen) ? (ti.n_kv != 0) : 1u;
    if (!counted) continue;
    const int q = ti.q0 + stage * C::BM + row;
    int vis_end = p.causal != kNoCausal ? min(p.N_k, q + 1 + p.causal) : p.N_k;  // keys < vis_end are visible
    if constexpr (C::kVarlen) vis_end = ti.coff != kNoCausal ? min(ti.len_k, q + 1 + ti.coff) : ti.len_k;
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < ti.n_kv; ++j) {
      if (!warp_wait(&bars.s_full[stage], s_par, wd, 0x30 + stage)) return;
      s_par ^= 1u;
      tc_fence_after();
      uint32_t s[C::BN];
#pragma unroll
      for (int c = 0; c < C::BN; c += 32) tmem_ld32(tS + c, s + c);
      tmem_ld_wait32(s);
#pragma unroll
      for (int c = 32; c < C::BN; c += 32) reg_fence32(s + c);

      const int lim = vis_end - (ti.j0 + j) * C::BN;  // columns c < lim are visible
      const bool need_mask = __any_sync(0xffffffffu, lim < C::BN);
      // Row max: three-input max over pairs, in kAcc independent chains (one
      // chain of BN dependent operations would put its whole latency on the
      // critical path).
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
        // O_s holds sum_{i<j} P_i V_i and no P.V is in flight (S_s(j) was
        // issued after P_s(j-1).V and its completion was just observed).
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
      // p = 2^(s*c - m) on pairs: packed FMA for the argument, ex2 on the
      // special-function unit, packed adds into kAcc/2 pair accumulators.
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
            e[k] = v0;
            e[k + 1] = v1;
            sum2[(k / 2) % (kAcc / 2)] = fadd2(sum2[(k / 2) % (kAcc / 2)], make_float2(v0, v1));
          }
          uint32_t pw[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) pw[k] = pack_bf16x2(e[2 * k], e[2 * k + 1]);
          tmem_st16(tS + c0 / 2, pw);
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
      const float sum = sum2[0].x + sum2[0].y;
      l_run += sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&bars.p_full[stage]);
    }
    // the row statistics: 1/l and LSE (natural log); l_run = 0 only for a row
    // that sees no key of the unit -- a split-KV unit, or bottom-right causal
    // with N_q > N_k: then O = 0 and LSE = -inf
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const float2 st = make_float2(inv_l, (m_run + __log2f(l_run)) * kLn2);
    if constexpr (C::kOwnEpilogue) {
      // three stages: this group writes its own rows once the last P.V is done
      if (!warp_wait(&bars.o_full[stage], tile_k & 1u, wd, 0x40 + stage)) return;
      tc_fence_after();
      store_stage<C>(p, ti, stage, st, tmem, lane_base, row, bars, tmO,
                     smem + C::kOffStage + (stage * 4 + wq) * C::kStoreBufBytes);
    } else {
      // two stages: hand them to the epilogue warpgroup
      if (!warp_wait(&bars.st_empty[stage], (tile_k & 1u) ^ 1u, wd, 0x34 + stage)) return;
      stats[stage * C::BM + row] = st;
      mbar_arrive_warp(&bars.st_full[stage]);
    }
  }
}

// The epilogue warpgroup (two stages): the row statistics come from the
// softmax groups through shared memory.
template <class C>
__device__ void tc_epilogue_role(const TcParams& p, uint32_t tmem, const Bars& bars,
                                 const float2* stats, const Watchdog& wd, const CUtensorMap* tmO, uint8_t* smem) {
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  uint32_t tile_k = 0;
  uint32_t counted = 0;  // empty work units (split-KV) take no pipeline phase
  UnitSource<C, false> src{p, bars, wd};
  for (int u = src.first(); u < p.n_units; u = src.next(u), tile_k += counted) {
    const TileInfo ti = tile_info<C>(p, u);
    counted = (C::kSplit || C::kVarlen) ? (ti.n_kv != 0) : 1u;
    if (!counted) continue;
#pragma unroll 1
    for (int s = 0; s < C::NST; ++s) {
      if (!warp_wait(&bars.o_full[s], tile_k & 1u, wd, 0x40 + s)) return;
      if (!warp_wait(&bars.st_full[s], tile_k & 1u, wd, 0x43 + s)) return;
      tc_fence_after();
      const float2 st = stats[s * C::BM + row];
      mbar_arrive_warp(&bars.st_empty[s]);
      store_stage<C>(p, ti, s, st, tmem, lane_base, row, bars, tmO, smem + C::kOffStage + wq * C::kStoreBufBytes);
    }
  }
}

// ------------------------------------------------------------------ kernel
template <class C>
__global__ void __launch_bounds__(512, 1)
fa_tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                 const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  Bars bars;
  constexpr int S = C::NST;
  bars.q_full = bar + 0 * S;
  bars.q_empty = bar + 1 * S;
  bars.s_full = bar + 2 * S;
  bars.p_full = bar + 3 * S;
  bars.o_full = bar + 4 * S;
  bars.o_empty = bar + 5 * S;
  bars.st_full = bar + 6 * S;
  bars.st_empty = bar + 7 * S;
  bars.kv_full = bar + 8 * S;
  bars.kv_empty = bar + 8 * S + C::NSLOT;
  bars.teardown = bar + 8 * S + 2 * C::NSLOT;
  bars.sq_unit = reinterpret_cast<volatile int*>(smem + C::kOffSched);
  bars.sq_full = reinterpret_cast<uint64_t*>(smem + C::kOffSched + 16);
  bars.sq_empty = bars.sq_full + kSchedDepth;
  float2* stats = reinterpret_cast<float2*>(smem + C::kOffStats);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], 4);  // one arrival per warp of a group
      mbar_init(&bars.o_full[s], 1);
      mbar_init(&bars.o_empty[s], 4);
      mbar_init(&bars.st_full[s], 4);
      mbar_init(&bars.st_empty[s], 4);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    mbar_init(&bars.teardown[0], 1);
    if constexpr (C::kVarlen)
      for (int e = 0; e < kSchedDepth; ++e) {
        mbar_init(&bars.sq_full[e], 1);
        mbar_init(&bars.sq_empty[e], kSchedConsumers);
      }
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
    if (warp == 12 && lane == 0) tc_load_role<C>(&tmQ, &tmK, &tmV, p, smem, bars, wd);
    if (warp == 13) tc_mma_role<C>(p, smem, tmem, bars, wd);
  } else if (wg == 2 && !C::kOwnEpilogue) {
    if constexpr (!C::kOwnEpilogue) {
      setmaxnreg_dec<C::kRegEpilogue>();
      tc_epilogue_role<C>(p, tmem, bars, stats, wd, &tmO, smem);
    }
  } else {
    setmaxnreg_inc<C::kRegSoftmax>();
    tc_softmax_role<C>(p, wg, tmem, bars, stats, wd, &tmO, smem);
  }
  // O stores still in flight finish before the CTA (and its shared memory)
  // goes away (a no-op for threads that issued none)
  if constexpr (C::kTmaStore)
    if (lane == 0) bulk_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if constexpr (C::kVarlen) {
    // every role of this CTA is done with the launch's counters; the last
    // CTA to get here zeroes them for the next launch that takes this slot
    if (threadIdx.x == 0) {
      unsigned int* ctr = p.err + 1 + 2 * p.sched_slot;
      __threadfence();
      if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
        atomicExch(ctr, 0u);
        atomicExch(ctr + 1, 0u);
      }
    }
  }
}

}  // namespace fa
