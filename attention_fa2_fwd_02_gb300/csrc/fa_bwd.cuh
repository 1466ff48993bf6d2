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
//  * fa_bwd_pre_kernel: delta and -LSE * log2(e) per query row into the
//    workspace (padded rows: delta = 0, -LSE = -inf, so their P is exactly 0),
//    and the fp32 dQ accumulator zeroed;
//  * fa_bwd_kernel: one work unit = one 128-key tile j of one (b, h).  K_j, V_j
//    stay in shared memory and dK_j, dV_j accumulate in tensor memory while
//    the unit walks the query tiles that see it (BM rows per step):
//    S^T = K_j Q_i^T and dP^T = V_j dO_i^T (lanes = keys), P^T and dS^T by two
//    compute warpgroups (each a half of the query columns), then
//    dV += P^T dO_i and dK += dS^T Q_i (A in tensor memory) and the step's dQ
//    contribution from dS^T staged in shared memory; dQ goes to one of two
//    tensor-memory buffers, so that its read-out overlaps the following
//    steps: the epilogue warps stage it in shared memory and add it into the
//    fp32 accumulator with TMA reductions (cp.reduce.async.bulk.tensor), one
//    per warp and 8 KB block -- per-element global reductions cost 6 % (d =
//    128) and 27 % (d = 64) of the whole backward.  At d = 128, S^T and dP^T
//    are double-buffered as well and the MMA warp issues step g's S^T and
//    dP^T before step g - 1's dV, dK and dQ, so that the tensor core works
//    while the compute warpgroups run (the step's dQ^T then lands in its own
//    S^T columns: see BwdCfg);
//  * fa_bwd_post_kernel: dQ = scale * accumulator in the output dtype.
//
// The dQ product: d = 128 uses 64-row query steps and computes dQ_i^T =
// K_j^T dS_i^T (M = head dim = 128 lanes, N = 64 queries), d = 64 uses
// 128-row steps and computes dQ_i = dS_i K_j (M = 128 queries, N = 64): either
// way one 64-column buffer, with M = 128 for the tensor core.
//
// Warp roles (512 threads): warpgroups 0 and 1 = compute (thread = key row =
// tensor-memory lane), warpgroup 2 = epilogue (dQ reductions; dK, dV stores
// at the end of a unit), warp 12 = TMA loads, warp 13 = MMA issue.  Tensor
// memory: d = 64: S^T (then P^T) | dP^T (then dS^T) | dV | dK | dQ x 2;
// d = 128: S^T x 2 (then P^T, then dQ^T) | dP^T x 2 (then dS^T) | dV | dK.
// Every wait is bounded (Watchdog).
#pragma once

#include "fa_ptx.cuh"

namespace fa {

struct BwdParams {
  int B, H, N_q, N_k;
  int H_kv, kv_group;     // K/V heads, query heads per K/V head (grouped-query attention)
  int causal;
  int causal_off;         // causal: key j visible to row i iff j <= i + causal_off
  float scale;            // softmax scale
  float scale_log2;       // scale * log2(e)
  int n_qt, n_kt;         // query tiles (BM rows) / key tiles (128)
  int N_qp;               // row pitch of the workspace vectors (N_q rounded up to 128)
  int n_units;            // B * H_kv * n_kt
  int head_group;         // K/V heads per schedule group (their dQ accumulator and Q, dO in L2)
  const float* nlse2;     // workspace: -LSE * log2(e) [B*H][N_qp] (-inf on padding)
  const float* delta;     // workspace: dO . O          [B*H][N_qp] (0 on padding)
  float* dq_acc;          // workspace: fp32 dQ / scale  [B*H][N_qp][D]
  void* dK;
  void* dV;
  long long dk_stride[3], dv_stride[3];  // elements: b, h, n
  unsigned int* err;
  unsigned long long timeout_ns;
  int d_qk, d_v;          // columns of dK and of dV to store (<= D; the columns of Q, K, V, dO
                          // past their extents load as zeros)
  int debug_flags;        // test hook: bit 0 = block 0 never delivers the second Q/dO step of its first unit
};

template <int D_>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr int BN = 128;             // keys per work unit (tensor-memory lanes)
  static constexpr int BM = D == 128 ? 64 : 128;  // query rows per step
  static constexpr bool kDqT = D == 128;     // dQ computed transposed (lanes = head dim)
  // d = 128: two S^T / dP^T buffers, so the tensor core computes the next
  // step's S^T and dP^T while the compute warpgroups work on this step's; a
  // step's dQ^T lands in its own S^T columns (issued after the dV product
  // that reads P^T there).  d = 64 (128-row steps) has no room for them.
  static constexpr bool kPipe = D == 128;
  static constexpr int kSBufs = kPipe ? 2 : 1;
  // Q/dO ring depth: step g + 1's S^T is issued right after step g - 1's
  // products free their slot, so the pipelined order needs a third slot to
  // keep the next Q/dO copy off its path
  static constexpr int NST = kPipe ? 3 : 2;
  static constexpr int kPanels = D / 64;     // 128-byte swizzle panels of 64 bf16 (head dim)
  static constexpr int kQPanels = BM / 64;   // panels of the dS^T tile (queries)
  static constexpr uint32_t kKVTileBytes = BN * D * 2;
  static constexpr uint32_t kKVPanelBytes = BN * 128;
  static constexpr uint32_t kQTileBytes = BM * D * 2;
  static constexpr uint32_t kQPanelBytes = BM * 128;
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kKVTileBytes;
  static constexpr uint32_t kOffQ = kOffV + kKVTileBytes;          // [NST]
  static constexpr uint32_t kOffdO = kOffQ + NST * kQTileBytes;    // [NST]
  static constexpr uint32_t kDsBytes = BN * BM * 2;
  static constexpr uint32_t kOffdS = kOffdO + NST * kQTileBytes;   // [kSBufs] dS^T [keys][queries]
  static constexpr uint32_t kOffDsEnd = kOffdS + kSBufs * kDsBytes;
  // The epilogue hands each step's dQ to the TMA engine as fp32 reduce-adds,
  // through 8 KB buffers per epilogue warp (two; one at d = 128, for shared
  // memory): d = 128 (dQ^T, lanes = head dims) 64 queries x the warp's 32
  // head dims, unswizzled; d = 64 (lanes = queries) the warp's 32 queries x
  // 64 head dims, as two 128-byte-swizzled 32 x 32 halves
  static constexpr uint32_t kDqStageBytes = 8192;
  static constexpr int kDqBufs = kPipe ? 1 : 2;
  static_assert(BM * 32 * 4 == kDqStageBytes || !kDqT, "d = 128 buffer: BM queries x 32 head dims");
  static_assert(32 * D * 4 == kDqStageBytes || kDqT, "d = 64 buffer: 32 queries x 64 head dims");
  static constexpr uint32_t kOffDqStage = (kOffDsEnd + 1023) / 1024 * 1024;
  static constexpr uint32_t kOffVec = kOffDqStage + 4 * kDqBufs * kDqStageBytes;  // [NST] -lse2[BM], delta[BM]
  static constexpr uint32_t kOffBar = kOffVec + NST * 2 * BM * 4;
  static constexpr int kNumBars = 13 + 2 * NST;  // + teardown
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + base alignment slack
  static constexpr uint32_t kThreads = 512;
  // tensor memory columns: S^T (P^T) and dP^T (dS^T) of buffer b, dV, dK,
  // and dQ buffer b (d = 128: dQ^T in the S^T columns of its step's buffer;
  // d = 64: two 64-column buffers of their own)
  __host__ __device__ static constexpr uint32_t col_s(uint32_t b) { return kPipe ? b * BM : 0; }
  __host__ __device__ static constexpr uint32_t col_dp(uint32_t b) { return kPipe ? (2 + b) * BM : BM; }
  static constexpr uint32_t kColdV = 2 * kSBufs * BM, kColdK = kColdV + D;
  __host__ __device__ static constexpr uint32_t col_dq(uint32_t b) { return kPipe ? col_s(b) : kColdK + D + b * 64; }
  static constexpr uint32_t kTmemCols = 512;
  // instruction descriptors (bf16 inputs, fp32 accumulators)
  static constexpr uint32_t kIdescS = make_idesc(1u, 128, BM, 0, 0);    // K-major A and B
  static constexpr uint32_t kIdescAcc = make_idesc(1u, 128, D, 0, 1);   // A in TMEM, B MN-major
  static constexpr uint32_t kIdescdQ = make_idesc(1u, 128, 64, 1, 1);   // A and B MN-major
  static constexpr uint32_t kKVBytes = 2 * kKVTileBytes;
  static constexpr uint32_t kStepBytes = 2 * kQTileBytes + 2 * BM * 4;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kColdK + D + (kPipe ? 0 : 128) == 512, "tensor memory layout");
  static_assert(!kPipe || BM == 64, "dQ^T (64 query columns) fills one S^T buffer");
  static_assert(kOffdS % 1024 == 0 && kDsBytes % 1024 == 0, "swizzled dS^T buffers");
};

struct BwdBars {
  uint64_t* kv_full;    // [1] K_j, V_j landed
  uint64_t* kv_empty;   // [1] unit's MMAs done with K_j, V_j
  uint64_t* s_full;     // [kSBufs] S^T, dP^T ready
  uint64_t* p_full;     // [kSBufs] P^T, dS^T written (256 arrivals)
  uint64_t* dkv_full;   // [1] unit's dK, dV complete
  uint64_t* dkv_empty;  // [1] dK, dV read out (128 arrivals)
  uint64_t* dq_full;    // [2] dQ buffer ready
  uint64_t* dq_empty;   // [2] dQ buffer read out (128 arrivals)
  uint64_t* q_full;     // [NST] Q_i, dO_i, -lse2_i, delta_i landed
  uint64_t* q_empty;    // [NST]
};

// Work unit u -> (b*H_kv + hk, key tile j).  K/V heads are taken in groups of
// head_group; inside a group the key tiles go in ascending j with the group's
// heads interleaved, so that concurrently running CTAs reduce into (and read
// Q, dO of) a few heads whose data stays in L2, and causal units come longest
// first (key tile j is seen by the query tiles from its diagonal on).  A unit
// walks, for each of the kv_group query heads that read K/V head hk, the
// query tiles i0 .. n_qt-1: step s is query head hk*kv_group + s / n_q, tile
// i0 + s % n_q.
struct BwdUnit {
  int b, hk, j, i0, n_q, n_steps;
};
struct BwdStep {
  int h, i;
  long long bh;  // b * H + h: the query head's rows of the workspace
};
template <class C>
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, int u) {
  BwdUnit w;
  const int BHk = p.B * p.H_kv;
  const int per_group = p.head_group * p.n_kt;
  const int g = u / per_group;
  const int rem = u - g * per_group;
  const int g0 = g * p.head_group;
  const int gh = min(p.head_group, BHk - g0);  // the last group may be smaller
  w.j = rem / gh;
  const int bhk = g0 + (rem - w.j * gh);
  w.b = bhk / p.H_kv;
  w.hk = bhk - w.b * p.H_kv;
  // first query tile holding a row that sees the tile's first key
  const int first_q = w.j * C::BN - p.causal_off;
  w.i0 = (p.causal && first_q > 0) ? first_q / C::BM : 0;
  w.n_q = w.i0 < p.n_qt ? p.n_qt - w.i0 : 0;
  w.n_steps = w.n_q * p.kv_group;
  return w;
}
__device__ __forceinline__ BwdStep bwd_step(const BwdParams& p, const BwdUnit& w, int s) {
  BwdStep t;
  const int g = s / w.n_q;
  t.i = w.i0 + (s - g * w.n_q);
  t.h = w.hk * p.kv_group + g;
  t.bh = static_cast<long long>(w.b) * p.H + t.h;
  return t;
}

// 1-D bulk copy global -> shared, completing on `bar` (16-byte aligned, size
// a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------- pre / post
// One warp per padded query row: delta = dO . O (fp32), nlse2 = -LSE * log2(e),
// dQ accumulator row zeroed.  Rows past N_q get delta 0 and nlse2 -inf.
struct BwdPreParams {
  int B, H, N_q, N_qp;
  const void* O;
  long long o_stride[3];
  const void* dO;
  long long do_stride[3];
  const float* LSE;
  long long lse_stride[3];
  float* nlse2;
  float* delta;
  float* dq_acc;
  int d_v;  // columns of O and dO (<= D)
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
  if (q < p.N_q && lane * PER < p.d_v) {  // (d_v is a multiple of 8: a lane's columns are all in or all out)
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
    // rows past N_q and rows that saw no key (LSE = -inf): -inf, so their P is 0
    const float lse = q < p.N_q ? p.LSE[b * p.lse_stride[0] + h * p.lse_stride[1] +
                                        static_cast<long long>(q) * p.lse_stride[2]]
                                : -INFINITY;
    p.nlse2[row] = lse == -INFINITY ? -INFINITY : -lse * 1.4426950408889634f;
  }
}

struct BwdPostParams {
  int B, H, N_q, N_qp;
  float scale;
  const float* dq_acc;
  void* dQ;
  long long dq_stride[3];
  int d_qk;  // columns of dQ (<= D)
};
template <typename T, int D>
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const __grid_constant__ BwdPostParams p) {
  constexpr int PER = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  const long long rows = static_cast<long long>(p.B) * p.H * p.N_q;
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  if (lane * PER >= p.d_qk) return;  // padded columns of the accumulator
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
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
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
      tma_load_4d(tmK, &bars.kv_full[0], smem + C::kOffK + pn * C::kKVPanelBytes, pn * 64, w.j * C::BN, w.hk, w.b,
                  pol_kv);
      tma_load_4d(tmV, &bars.kv_full[0], smem + C::kOffV + pn * C::kKVPanelBytes, pn * 64, w.j * C::BN, w.hk, w.b,
                  pol_kv);
    }
    ++kv_armed;
    ++ku;
    for (int s = 0; ok && s < w.n_steps; ++s, ++gs) {
      const BwdStep t = bwd_step(p, w, s);
      const int i = t.i;
      const uint32_t st = gs % C::NST;
      if (!(ok = mbar_wait(&bars.q_empty[st], ((gs / C::NST) & 1u) ^ 1u, wd, 0x61))) break;
      // test hook (host-set flag): this step never arrives, so the bounded
      // waits on it run out; it is not armed, so the drain below skips it
      if ((p.debug_flags & 1) && blockIdx.x == 0 && gs == 1) continue;
      mbar_arrive_expect_tx(&bars.q_full[st], C::kStepBytes);
#pragma unroll
      for (int pn = 0; pn < C::kPanels; ++pn) {
        tma_load_4d(tmQ, &bars.q_full[st], smem + C::kOffQ + st * C::kQTileBytes + pn * C::kQPanelBytes, pn * 64,
                    i * C::BM, t.h, w.b, pol_q);
        tma_load_4d(tmdO, &bars.q_full[st], smem + C::kOffdO + st * C::kQTileBytes + pn * C::kQPanelBytes,
                    pn * 64, i * C::BM, t.h, w.b, pol_q);
      }
      const long long vrow = t.bh * p.N_qp + i * C::BM;
      uint8_t* vec = smem + C::kOffVec + st * 2 * C::BM * 4;
      bulk_load(vec, p.nlse2 + vrow, C::BM * 4, &bars.q_full[st]);
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

// k-step kk (16 elements of K) of a K-major operand: a bf16 tile whose rows are
// M or N, K along the 128-byte swizzle panels.
template <uint32_t kPanelBytes>
__device__ __forceinline__ uint32_t kmajor_off(int kk) {
  const uint32_t byte = kk * 32;
  return ((byte / 128) * kPanelBytes + byte % 128) >> 4;
}

// Column (within the S^T or dP^T region) of the bf16 pairs of queries
// 16 kk .. 16 kk + 15: the compute warpgroup owning them stores them in the
// first half of its own columns.
template <class C>
__device__ __forceinline__ uint32_t pcol(int kk) {
  constexpr int kCols = C::BM / 2;
  return (16 * kk / kCols) * kCols + (16 * kk % kCols) / 2;
}

template <class C>
__device__ void bwd_mma_role(const BwdParams& p, uint8_t* smem, uint32_t tmem, const BwdBars& bars,
                             const Watchdog& wd, uint64_t* teardown) {
  const uint32_t k_addr = smem_u32(smem + C::kOffK);
  const uint32_t v_addr = smem_u32(smem + C::kOffV);
  uint32_t ku = 0, gs = 0;
  bool ok = true;
  // S^T(g) = K Q_g^T and dP^T(g) = V dO_g^T into buffer g mod kSBufs.  The
  // buffer's previous contents: P^T / dS^T of step g - kSBufs, whose dV and
  // dK products were issued before (in-order execution), and (d = 128) its
  // dQ^T, which the epilogue must have read out.
  auto issue_s = [&](uint32_t g) -> bool {
    const uint32_t st = g % C::NST, b = g % C::kSBufs;
    if (!bwd_warp_wait(&bars.q_full[st], (g / C::NST) & 1u, wd, 0x63)) return false;
    if (C::kPipe && g >= 2 && !bwd_warp_wait(&bars.dq_empty[b], ((g >> 1) - 1) & 1u, wd, 0x64)) return false;
    tc_fence_after();
    if (elect_one()) {
      const uint32_t q_addr = smem_u32(smem + C::kOffQ + st * C::kQTileBytes);
      const uint32_t do_addr = smem_u32(smem + C::kOffdO + st * C::kQTileBytes);
      const uint64_t ak = sdesc_sw128<16, 1024>(k_addr), av = sdesc_sw128<16, 1024>(v_addr);
      const uint64_t bq = sdesc_sw128<16, 1024>(q_addr), bdo = sdesc_sw128<16, 1024>(do_addr);
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk)
        mma_ss<false>(tmem + C::col_s(b), ak + kmajor_off<C::kKVPanelBytes>(kk), bq + kmajor_off<C::kQPanelBytes>(kk),
                      C::kIdescS, kk > 0);
#pragma unroll
      for (int kk = 0; kk < C::D / 16; ++kk)
        mma_ss<false>(tmem + C::col_dp(b), av + kmajor_off<C::kKVPanelBytes>(kk),
                      bdo + kmajor_off<C::kQPanelBytes>(kk), C::kIdescS, kk > 0);
      tc_commit(&bars.s_full[b]);
    }
    __syncwarp();
    return true;
  };
  // dV += P^T dO_g, dK += dS^T Q_g and dQ of step g, once the compute
  // warpgroups have written P^T(g) and dS^T(g)
  auto finish = [&](uint32_t g, bool first, bool last) -> bool {
    const uint32_t st = g % C::NST, b = g % C::kSBufs, qb = g & 1u;
    if (!bwd_warp_wait(&bars.p_full[b], (g / C::kSBufs) & 1u, wd, 0x65)) return false;
    // the first accumulation of a unit overwrites dK, dV: the previous
    // unit's must have been read out
    if (first && ku > 0 && !bwd_warp_wait(&bars.dkv_empty[0], (ku - 1) & 1u, wd, 0x66)) return false;
    // d = 64: the dQ buffer of two steps ago must have been read out
    if (!C::kPipe && g >= 2 && !bwd_warp_wait(&bars.dq_empty[qb], ((g >> 1) - 1) & 1u, wd, 0x64)) return false;
    tc_fence_after();
    if (elect_one()) {
      const uint32_t q_addr = smem_u32(smem + C::kOffQ + st * C::kQTileBytes);
      const uint32_t do_addr = smem_u32(smem + C::kOffdO + st * C::kQTileBytes);
      // dV += P^T dO_g and dK += dS^T Q_g: A in tensor memory (bf16 pairs),
      // B MN-major (head dim contiguous, k = query rows in 16-row steps)
      const uint64_t bdo = sdesc_sw128<C::kQPanelBytes, 1024>(do_addr);
      const uint64_t bq = sdesc_sw128<C::kQPanelBytes, 1024>(q_addr);
#pragma unroll
      for (int kk = 0; kk < C::BM / 16; ++kk)
        mma_ts<false>(tmem + C::kColdV, tmem + C::col_s(b) + pcol<C>(kk), bdo + ((kk * 16 * 128) >> 4), C::kIdescAcc,
                      (!first || kk > 0) ? 1u : 0u);
      auto issue_dk = [&]() {
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_ts<false>(tmem + C::kColdK, tmem + C::col_dp(b) + pcol<C>(kk), bq + ((kk * 16 * 128) >> 4),
                        C::kIdescAcc, (!first || kk > 0) ? 1u : 0u);
      };
      // dQ over the keys (k = 16-key steps of 16 rows x 128 bytes):
      //  d = 128: dQ_g^T = K_j^T dS_g^T, A = K_j MN-major (head dim
      //           contiguous), B = dS^T MN-major (queries contiguous);
      //  d = 64:  dQ_g = dS_g K_j, A = dS^T MN-major, B = K_j MN-major.
      // Without a causal mask dQ goes before dK (it only has to follow dV,
      // which reads P^T where dQ^T lands at d = 128), so that the epilogue
      // reads it out sooner: measured +8.5 % on the non-causal backward, but
      // -3 % on the causal one (also with dK first on a unit's last step), so
      // causal problems keep dK first.
      const bool dq_first = !p.causal;
      if (!dq_first) issue_dk();
      const uint32_t ds_addr = smem_u32(smem + C::kOffdS + b * C::kDsBytes);
      const uint64_t dsd = sdesc_sw128<C::BN * 128, 1024>(ds_addr);
      const uint64_t kd = sdesc_sw128<C::kKVPanelBytes, 1024>(k_addr);
      const uint64_t a0 = C::kDqT ? kd : dsd, b0 = C::kDqT ? dsd : kd;
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_ss<false>(tmem + C::col_dq(qb), a0 + ((kk * 16 * 128) >> 4), b0 + ((kk * 16 * 128) >> 4), C::kIdescdQ,
                      kk > 0 ? 1u : 0u);
      tc_commit(&bars.dq_full[qb]);
      if (dq_first) issue_dk();
      tc_commit(&bars.q_empty[st]);
      if (last) {
        tc_commit(&bars.dkv_full[0]);
        tc_commit(&bars.kv_empty[0]);
      }
    }
    __syncwarp();
    return true;
  };
  for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    if (w.n_steps == 0) continue;
    if (!(ok = bwd_warp_wait(&bars.kv_full[0], ku & 1u, wd, 0x62))) break;
    const uint32_t g0 = gs;
    for (int s = 0; ok && s < w.n_steps; ++s, ++gs) {
      if (!(ok = issue_s(gs))) break;
      if constexpr (C::kPipe) {
        // the previous step's products after this step's S^T, dP^T: the
        // tensor core works on them while the compute warpgroups run step s
        if (s > 0) ok = finish(gs - 1, s == 1, false);
      } else {
        ok = finish(gs, s == 0, s == w.n_steps - 1);
      }
    }
    if (C::kPipe && ok) ok = finish(gs - 1, gs - 1 == g0, true);
    ++ku;
  }
  if (!ok) {
    if (elect_one()) tc_commit(teardown);
    __syncwarp();
    mbar_drain(teardown, 0, 100000000ull);
  }
}

// Two warpgroups (cg = 0, 1), each a half of the step's query columns; the
// bf16 P^T / dS^T of warpgroup cg sit at columns cg*kCols + (query % kCols)/2.
template <class C>
__device__ void bwd_compute_role(const BwdParams& p, uint8_t* smem, uint32_t tmem, const BwdBars& bars,
                                 const Watchdog& wd, int cg) {
  constexpr int kCols = C::BM / 2;  // query columns per warpgroup: 32 or 64
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int r = wq * 32 + lane;  // key row of the tile = tensor-memory lane
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  uint8_t* const ds_row0 = smem + C::kOffdS + r * 128;
  const float sc = p.scale_log2;
  const float2 sc2 = make_float2(sc, sc);
  uint32_t gs = 0;
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    const int key = w.j * C::BN + r;
    const bool key_ok = key < p.N_k;
    for (int s = 0; s < w.n_steps; ++s, ++gs) {
      const int q0 = bwd_step(p, w, s).i * C::BM + cg * kCols;  // first query of this warpgroup's columns
      const uint32_t st = gs % C::NST;
      const float* nl2 = reinterpret_cast<const float*>(smem + C::kOffVec + st * 2 * C::BM * 4) + cg * kCols;
      const float* dlt = nl2 + C::BM;
      const uint32_t b = gs % C::kSBufs;
      const uint32_t tS = tmem + lane_base + C::col_s(b);
      const uint32_t tdP = tmem + lane_base + C::col_dp(b);
      uint8_t* const ds_row = ds_row0 + b * C::kDsBytes;
      if (!bwd_warp_wait(&bars.s_full[b], (gs / C::kSBufs) & 1u, wd, 0x67)) return;
      tc_fence_after();
      // per-element masking only where needed: the key tail and tiles that
      // reach above the diagonal (query tails have -lse2 = -inf)
      const bool need_mask = __any_sync(0xffffffffu, !key_ok || (p.causal && key > q0 + p.causal_off));
#pragma unroll 1
      for (int c0 = 0; c0 < kCols; c0 += 32) {
        uint32_t sv[32], dpv[32];
        tmem_ld32(tS + cg * kCols + c0, sv);
        tmem_ld32(tdP + cg * kCols + c0, dpv);
        tmem_ld_wait32(sv);
        reg_fence32(dpv);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          const float4 l2 = *reinterpret_cast<const float4*>(nl2 + c0 + k);
          const float4 dl = *reinterpret_cast<const float4*>(dlt + c0 + k);
#pragma unroll
          for (int h = 0; h < 4; h += 2) {
            const int c = c0 + k + h;
            const float2 x = ffma2(make_float2(__uint_as_float(sv[k + h]), __uint_as_float(sv[k + h + 1])), sc2,
                                   h ? make_float2(l2.z, l2.w) : make_float2(l2.x, l2.y));
            float p0 = ex2(x.x), p1 = ex2(x.y);
            if (need_mask) {
              if (!key_ok || (p.causal && key > q0 + c + p.causal_off)) p0 = 0.f;
              if (!key_ok || (p.causal && key > q0 + c + 1 + p.causal_off)) p1 = 0.f;
            }
            const float2 g = fadd2(make_float2(__uint_as_float(dpv[k + h]), __uint_as_float(dpv[k + h + 1])),
                                   h ? make_float2(-dl.z, -dl.w) : make_float2(-dl.x, -dl.y));
            const float2 ds = fmul2(make_float2(p0, p1), g);
            pw[(k + h) / 2] = pack_bf16x2(p0, p1);
            dw[(k + h) / 2] = pack_bf16x2(ds.x, ds.y);
          }
        }
        // P^T and dS^T (bf16 pairs) go into the first half of this
        // warpgroup's own S^T / dP^T columns: column c0/2 + k < c0 + 32, all
        // read by this thread already (the MMA warp addresses each 16-query
        // k-step there)
        tmem_st16(tS + cg * kCols + c0 / 2, pw);
        tmem_st16(tdP + cg * kCols + c0 / 2, dw);
        // dS^T row r, queries of this chunk, into the 128-byte-swizzled panel
        // layout (64 queries per panel, 8-row groups of 1024 bytes)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int qc = cg * kCols + c0 + 8 * t;  // first query (of the step) of the 16-byte chunk
          uint8_t* panel = ds_row + (qc / 64) * (C::BN * 128);
          const int chunk = ((qc % 64) / 8) ^ (r & 7);
          *reinterpret_cast<uint4*>(panel + chunk * 16) =
              make_uint4(dw[4 * t], dw[4 * t + 1], dw[4 * t + 2], dw[4 * t + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // dS^T stores -> the tensor core's reads
      tc_fence_before();
      mbar_arrive(&bars.p_full[b]);
    }
  }
}

template <class C>
__device__ void bwd_epilogue_role(const CUtensorMap* tmDq, const BwdParams& p, uint8_t* smem, uint32_t tmem,
                                  const BwdBars& bars, const Watchdog& wd) {
  const int wq = (threadIdx.x / 32) & 3;
  const int lane = threadIdx.x & 31;
  const int r = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  uint8_t* dq_stage = smem + C::kOffDqStage + wq * C::kDqBufs * C::kDqStageBytes;  // this warp's buffers
  uint32_t n_red = 0;                                                     // reductions issued
  uint32_t ku = 0, gs = 0;
  auto run = [&]() {
  for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
    const BwdUnit w = bwd_unit<C>(p, u);
    const int key = w.j * C::BN + r;
    __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(p.dK) + w.b * p.dk_stride[0] +
                            w.hk * p.dk_stride[1] + static_cast<long long>(key) * p.dk_stride[2];
    __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(p.dV) + w.b * p.dv_stride[0] +
                            w.hk * p.dv_stride[1] + static_cast<long long>(key) * p.dv_stride[2];
    if (w.n_steps == 0) {  // keys no query sees: zero gradients
      if (key < p.N_k)
        for (int c = 0; c < C::D; c += 8) {
          if (c < p.d_qk) *reinterpret_cast<uint4*>(dk_row + c) = make_uint4(0, 0, 0, 0);
          if (c < p.d_v) *reinterpret_cast<uint4*>(dv_row + c) = make_uint4(0, 0, 0, 0);
        }
      continue;
    }
    for (int s = 0; s < w.n_steps; ++s, ++gs) {
      const BwdStep t = bwd_step(p, w, s);
      const uint32_t qb = gs & 1u;
      const int q0 = t.i * C::BM;
      if (!bwd_warp_wait(&bars.dq_full[qb], (gs >> 1) & 1u, wd, 0x68)) return;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tmem + lane_base + C::col_dq(qb), v);
      tmem_ld32(tmem + lane_base + C::col_dq(qb) + 32, v + 32);
      tmem_ld_wait32(v);
      reg_fence32(v + 32);
      tc_fence_before();
      mbar_arrive(&bars.dq_empty[qb]);  // the values are in registers now
      if constexpr (!C::kDqT) {
        // lane r = query row of the step, columns = the 64 head dims: the
        // warp's 32 x 64 block in two 32 x 32 halves, each row a 128-byte
        // swizzle row (16-byte chunk i at i ^ (row mod 8): conflict-free
        // quarter-warps), and one lane adds them with two TMA reductions
        static_assert(C::kDqBufs == 2, "d = 64: two staging buffers per warp");
        uint8_t* buf = dq_stage + (n_red & 1u) * C::kDqStageBytes;
        if (n_red >= 2) {  // the reductions that last read this buffer
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(buf + h * 4096 + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                make_float4(__uint_as_float(v[32 * h + 4 * i]), __uint_as_float(v[32 * h + 4 * i + 1]),
                            __uint_as_float(v[32 * h + 4 * i + 2]), __uint_as_float(v[32 * h + 4 * i + 3]));
        fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(tmDq, buf, 0, q0 + wq * 32, static_cast<int>(t.bh));
          tma_reduce_add_3d(tmDq, buf + 4096, 32, q0 + wq * 32, static_cast<int>(t.bh));
          bulk_commit();
        }
        ++n_red;
      } else {
        // lane r = head-dim index, columns = the step's 64 queries: the warp's
        // 64 x 32 block goes through its shared-memory buffer (row = query,
        // 32 consecutive head dims: every store instruction covers one
        // 128-byte row) and one lane adds it into the accumulator with a TMA
        // reduction
        static_assert(C::kDqBufs == 1, "d = 128: one staging buffer per warp");
        float* buf = reinterpret_cast<float*>(dq_stage);
        if (n_red >= 1) {  // the reduction that last read this buffer
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int c = 0; c < 64; ++c) buf[c * 32 + lane] = __uint_as_float(v[c]);
        fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(tmDq, buf, wq * 32, q0, static_cast<int>(t.bh));
          bulk_commit();
        }
        ++n_red;
      }
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
          if (c + k < p.d_v)
            *reinterpret_cast<uint4*>(dv_row + c + k) =
                make_uint4(pack_bf16x2(__uint_as_float(v[k]), __uint_as_float(v[k + 1])),
                           pack_bf16x2(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])),
                           pack_bf16x2(__uint_as_float(v[k + 4]), __uint_as_float(v[k + 5])),
                           pack_bf16x2(__uint_as_float(v[k + 6]), __uint_as_float(v[k + 7])));
          if (c + k < p.d_qk)
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
  };
  run();
  // the reductions must have read their buffers (and landed) before the
  // CTA's shared memory goes away and before the dQ conversion reads the
  // accumulator, on every exit path
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

template <class C>
__global__ void __launch_bounds__(512, 1)
fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tmDq) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  BwdBars bars;
  bars.kv_full = bar + 0;
  bars.kv_empty = bar + 1;
  bars.s_full = bar + 2;     // [2]
  bars.p_full = bar + 4;     // [2]
  bars.dkv_full = bar + 6;
  bars.dkv_empty = bar + 7;
  bars.dq_full = bar + 8;    // [2]
  bars.dq_empty = bar + 10;  // [2]
  bars.q_full = bar + 12;
  bars.q_empty = bar + 12 + C::NST;
  uint64_t* teardown = bar + 12 + 2 * C::NST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full[0], 1);
    mbar_init(&bars.kv_empty[0], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.p_full[b], 256);
    }
    mbar_init(&bars.dkv_full[0], 1);
    mbar_init(&bars.dkv_empty[0], 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.dq_full[b], 1);
      mbar_init(&bars.dq_empty[b], 128);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bars.q_full[s], 1);
      mbar_init(&bars.q_empty[s], 1);
    }
    mbar_init(teardown, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmdO);
    prefetch_tensormap(&tmDq);
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
  // register split (setmaxnreg, per warpgroup): the shares must add up to
  // the 4 x 128 registers per thread the block was launched with
  constexpr uint32_t kRegCompute = 144, kRegEpilogue = 112, kRegProducer = 112;
  static_assert(2 * kRegCompute + kRegEpilogue + kRegProducer == 4 * 128, "register split");
  if (warp < 8) {
    setmaxnreg_inc<kRegCompute>();
    bwd_compute_role<C>(p, smem, tmem, bars, wd, warp / 4);
  } else if (warp < 12) {
    setmaxnreg_dec<kRegEpilogue>();
    bwd_epilogue_role<C>(&tmDq, p, smem, tmem, bars, wd);
  } else {
    setmaxnreg_dec<kRegProducer>();
    if (warp == 12) {
      if (lane == 0) bwd_load_role<C>(&tmQ, &tmK, &tmV, &tmdO, p, smem, bars, wd);
    } else if (warp == 13) {
      bwd_mma_role<C>(p, smem, tmem, bars, wd, teardown);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
