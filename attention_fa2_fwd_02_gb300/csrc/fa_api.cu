// fa_api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument
// validation, TMA descriptor encoding, kernel selection and launch, and the
// device error word behind fa_check().  Host-side only, apart from the
// small-head kernel instantiations, which live here too.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "fa.h"
#include "fa_combine.cuh"
#include "fa_launch.h"
#include "fa_axial_block.cuh"
#include "fa_small.cuh"
#include "fa_small_mma.cuh"
#include "fa_vt.cuh"

namespace fa {
// [0]: raised (atomicOr) by any kernel of this library whose bounded wait
// expires.  [1 + 2 s], [2 + 2 s]: the work-unit counters of packed-batch
// launches (scheduler slot s: units taken, CTAs done; zero between launches).
__device__ unsigned int g_err_word[1 + 2 * kSchedSlots];
}  // namespace fa

namespace {

using namespace fa;

thread_local std::string t_last_error;

fa_status_t fail(fa_status_t st, const std::string& msg) {
  t_last_error = msg;
  return st;
}

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

std::atomic<unsigned long long> g_timeout_ns{1000000000ull};
std::atomic<int> g_debug_flags{0};
std::atomic<unsigned int> g_sched_next{0};  // next scheduler slot of a packed-batch launch

struct DevState {
  bool ready = false;
  int device = 0;
  int sm_count = 0;
  unsigned int* err = nullptr;
  bool small_attr[2][2] = {{false, false}, {false, false}};  // [bf16/fp32][d16/d32] opt-in set
  bool axial_attr = false;                                   // fused axial block opt-in set
};
std::mutex g_mu;
DevState g_dev[kMaxDevices];

fa_status_t device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("cudaGetDevice", e));
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_CUDA, "device ordinal out of range");
  // Bind the device's primary context to the calling thread: the tensor maps
  // are encoded with a driver call, which needs a current context, and a
  // thread that has made no runtime call yet (an autograd worker, say) has
  // none.
  if ((e = cudaSetDevice(dev)) != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("cudaSetDevice", e));
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& s = g_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail(FA_ERR_CUDA, cuda_msg("cudaDeviceGetAttribute", e));
    if (major != 10 || minor != 3)
      return fail(FA_ERR_UNSUPPORTED, "libfa.so is built for sm_103a (GB300); device has compute capability " +
                                          std::to_string(major) + "." + std::to_string(minor));
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_err_word)) != cudaSuccess)
      return fail(FA_ERR_CUDA, cuda_msg("cudaGetSymbolAddress(error word)", e));
    s.err = static_cast<unsigned int*>(p);
    s.device = dev;
    s.ready = true;
  }
  *out = &s;
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

enum class Path { kTensorCore, kSmall };

bool tensor_ok(const fa_tensor_t& t) { return t.ptr != nullptr && t.stride[3] == 1; }
long long kv_heads(const fa_problem_t& pb) { return pb.H_kv > 0 ? pb.H_kv : pb.H; }

long long v_dim(const fa_problem_t& pb) { return pb.Dv > 0 ? pb.Dv : pb.d; }
// Tensor-core tile width for head dims d (Q, K) and dv (V, O): 64, 128 or
// 256 columns (256: the bf16 kernel for head dims above 128); columns past d
// or dv are loaded as zeros.
int tc_tile_dim(long long d, long long dv) {
  return (d > 128 || dv > 128) ? 256 : ((d > 64 || dv > 64) ? 128 : 64);
}

// Validate one problem and choose its kernel (tensor_core_only: never the
// small-head path).
fa_status_t validate(fa_dtype_t dtype, const fa_problem_t& pb, int idx, Path* path,
                     bool tensor_core_only = false) {
  const std::string at = "problem " + std::to_string(idx) + ": ";
  if (dtype != FA_BF16 && dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, at + "unknown dtype");
  if (pb.B <= 0 || pb.H <= 0 || pb.N_q <= 0 || pb.N_k <= 0 || pb.d <= 0)
    return fail(FA_ERR_INVALID_ARG, at + "B, H, N_q, N_k and d must all be >= 1");
  if (!tensor_ok(pb.Q) || !tensor_ok(pb.K) || !tensor_ok(pb.V) || !tensor_ok(pb.O))
    return fail(FA_ERR_INVALID_ARG, at + "Q, K, V, O need a non-null pointer and stride[3] == 1");
  if (!std::isfinite(pb.scale)) return fail(FA_ERR_INVALID_ARG, at + "scale must be finite");
  if (pb.H_kv < 0 || (pb.H_kv > 0 && pb.H % pb.H_kv != 0))
    return fail(FA_ERR_INVALID_ARG, at + "H_kv must divide H (0 = H)");
  if (pb.is_causal < 0 || pb.is_causal > 2)
    return fail(FA_ERR_INVALID_ARG, at + "is_causal must be 0, 1 (top-left) or 2 (bottom-right)");
  if (pb.LSE && (pb.lse_stride[0] < 0 || pb.lse_stride[1] < 0 || pb.lse_stride[2] < 0))
    return fail(FA_ERR_UNSUPPORTED, at + "negative LSE strides are not supported");
  const fa_tensor_t* ts[4] = {&pb.Q, &pb.K, &pb.V, &pb.O};
  for (auto* t : ts)
    for (int i = 0; i < 3; ++i)
      if (t->stride[i] < 0) return fail(FA_ERR_UNSUPPORTED, at + "negative strides are not supported");
  if (pb.N_q >= (1ll << 31) || pb.N_k >= (1ll << 31) || pb.B >= (1ll << 31) || pb.H >= (1ll << 31))
    return fail(FA_ERR_UNSUPPORTED, at + "sizes must be below 2^31");
  if (pb.Dv < 0) return fail(FA_ERR_INVALID_ARG, at + "Dv must be >= 0 (0 = d)");
  const long long dv = v_dim(pb);
  if ((pb.d == 16 || pb.d == 32) && dv == pb.d && !tensor_core_only) {
    const long long items = pb.B * pb.H * ((pb.N_q + 31) / 32);
    if (items >= (1ll << 40)) return fail(FA_ERR_UNSUPPORTED, at + "too many query blocks");
    *path = Path::kSmall;
    return FA_OK;
  }
  const long long E = dtype == FA_FP32 ? 4 : 2;
  const long long max_dim = dtype == FA_FP32 ? 128 : 256;
  if (pb.d > max_dim || dv > max_dim || (pb.d * E) % 16 != 0 || (dv * E) % 16 != 0)
    return fail(FA_ERR_UNSUPPORTED, at + "head dims d = " + std::to_string(pb.d) + ", Dv = " + std::to_string(dv) +
                                        " not supported (up to 256 in bf16, 128 in fp32, rows of a multiple of 16 "
                                        "bytes; or d = Dv in {16, 32} on the small-head path)");
  for (auto* t : ts) {
    if (reinterpret_cast<uintptr_t>(t->ptr) % 16 != 0)
      return fail(FA_ERR_UNSUPPORTED, at + "tensor-core path needs 16-byte aligned base pointers");
    for (int i = 0; i < 3; ++i)
      if ((t->stride[i] * E) % 16 != 0)
        return fail(FA_ERR_UNSUPPORTED, at + "tensor-core path needs strides that are multiples of 16 bytes");
  }
  const long long tiles = pb.B * pb.H * ((pb.N_q + 127) / 128);  // (128-row tiles of the wide kernel)
  if (tiles >= (1ll << 31)) return fail(FA_ERR_UNSUPPORTED, at + "too many query tiles");
  *path = Path::kTensorCore;
  return FA_OK;
}

fa_status_t make_map(CUtensorMap* map, const fa_tensor_t& t, bool fp32, long long B, long long H, long long N,
                     long long d, int box_rows, const char* name) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const long long E = fp32 ? 4 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(t.stride[2] * E), (cuuint64_t)(t.stride[1] * E),
                           (cuuint64_t)(t.stride[0] * E)};
  cuuint32_t box[4] = {(cuuint32_t)tc_box_inner(fp32), (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  // fp32 inputs go to the tf32 tensor cores: a tf32-typed map makes the copy
  // round each value to tf32 (nearest, ties to even) on its way to shared memory
  CUresult r = enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_TFLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.ptr, dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FA_ERR_UNSUPPORTED, std::string("cuTensorMapEncodeTiled rejected the layout of ") + name +
                                        " (CUresult " + std::to_string((int)r) + ")");
  return FA_OK;
}

// Split-KV workspace (caller-owned): fp32 partial O [n_split][B*H*N_q][d],
// then fp32 partial LSE [n_split][B*H*N_q], each part 256-byte aligned.
struct SplitWs {
  float* o = nullptr;
  float* lse = nullptr;
};
size_t split_ws_bytes(long long B, long long H, long long N_q, long long d, int n_split) {
  const size_t rows = static_cast<size_t>(B) * H * N_q;
  const size_t o = (static_cast<size_t>(n_split) * rows * d * 4 + 255) & ~size_t(255);
  const size_t l = (static_cast<size_t>(n_split) * rows * 4 + 255) & ~size_t(255);
  return o + l;
}
SplitWs split_ws_layout(void* ws, long long B, long long H, long long N_q, long long d, int n_split) {
  const size_t rows = static_cast<size_t>(B) * H * N_q;
  const size_t o = (static_cast<size_t>(n_split) * rows * d * 4 + 255) & ~size_t(255);
  SplitWs w;
  w.o = static_cast<float*>(ws);
  w.lse = reinterpret_cast<float*>(static_cast<char*>(ws) + o);
  return w;
}

// V^T workspace of the fp32 tensor-core path (fa_vt.cuh): [B * H_kv][Dv][ldk]
// fp32, ldk = N_k rounded up to 32.
long long vt_ldk(long long N_k) { return (N_k + 31) / 32 * 32; }
size_t vt_ws_bytes(const fa_problem_t& pb) {
  return static_cast<size_t>(pb.B) * kv_heads(pb) * v_dim(pb) * vt_ldk(pb.N_k) * 4;
}
// A problem takes the V^T pass when it runs on the tf32 tensor cores and each
// V tile is read by at least two query tiles (query blocks x the query heads
// of a K/V head): the pass then saves at least one in-kernel transpose per
// V tile.
bool wants_vt(fa_dtype_t dtype, const fa_problem_t& pb, Path path) {
  if (dtype != FA_FP32 || path != Path::kTensorCore) return false;
  const long long uses = (pb.N_q + kWideQueryTile - 1) / kWideQueryTile * (pb.H / kv_heads(pb));
  return uses >= 2;
}

fa_status_t make_vt_map(CUtensorMap* map, const float* vt, const fa_problem_t& pb, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const long long ldk = vt_ldk(pb.N_k), dv = v_dim(pb);
  cuuint64_t dims[4] = {(cuuint64_t)pb.N_k, (cuuint64_t)dv, (cuuint64_t)kv_heads(pb), (cuuint64_t)pb.B};
  cuuint64_t strides[3] = {(cuuint64_t)(ldk * 4), (cuuint64_t)(dv * ldk * 4), (cuuint64_t)(kv_heads(pb) * dv * ldk * 4)};
  cuuint32_t box[4] = {32, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_TFLOAT32, 4, const_cast<float*>(vt), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the V^T workspace (CUresult " +
                                        std::to_string((int)r) + ")");
  return FA_OK;
}

// vt: the V^T workspace (fp32, unsplit) or null (V tiles transposed in the kernel).
fa_status_t launch_tensor_core(fa_dtype_t dtype, const fa_problem_t& pb, const DevState& ds, cudaStream_t stream,
                               int n_split = 1, SplitWs ws = SplitWs{}, float* vt = nullptr) {
  const bool fp32 = dtype == FA_FP32;
  const int dv = static_cast<int>(v_dim(pb));
  const int d = tc_tile_dim(pb.d, dv);  // the kernel's tile width
  if (n_split > 1 && (pb.d != d || dv != d || d == 256))
    return fail(FA_ERR_UNSUPPORTED, "split-KV needs d = Dv in {64, 128}");
  // the single-stage kernel (fa_tc_wide.cuh): bf16 tiles of 256 columns and
  // every fp32 problem (split or not)
  const bool wide = d == 256 || fp32;
  const int stages = tc_stages(fp32, d, pb.is_causal != 0, n_split > 1);  // (two-stage kernel)
  const int bn = wide ? kWideKeyTile : tc_key_tile(stages);
  const int bm = wide ? kWideQueryTile : tc_tile_rows(stages);  // query rows of a CTA tile
  TcLaunch L;
  fa_status_t st;
  if ((st = make_map(&L.tmQ, pb.Q, fp32, pb.B, pb.H, pb.N_q, pb.d, 128, "Q")) != FA_OK) return st;
  if ((st = make_map(&L.tmK, pb.K, fp32, pb.B, kv_heads(pb), pb.N_k, pb.d, bn, "K")) != FA_OK) return st;
  if (vt) {
    if (!fp32 || n_split > 1) return fail(FA_ERR_UNSUPPORTED, "the V^T pass serves the unsplit fp32 path");
    if ((st = make_vt_map(&L.tmV, vt, pb, d)) != FA_OK) return st;
  } else if ((st = make_map(&L.tmV, pb.V, fp32, pb.B, kv_heads(pb), pb.N_k, dv, bn, "V")) != FA_OK) {
    return st;
  }
  if (n_split == 1 && (st = make_map(&L.tmO, pb.O, fp32, pb.B, pb.H, pb.N_q, dv, 32, "O")) != FA_OK)
    return st;
  TcParams& p = L.p;
  p.B = (int)pb.B;
  p.H = (int)pb.H;
  p.N_q = (int)pb.N_q;
  p.N_k = (int)pb.N_k;
  p.causal = pb.is_causal == 0 ? kNoCausal : (pb.is_causal == 2 ? (int)(pb.N_k - pb.N_q) : 0);
  p.scale_log2 = static_cast<float>(static_cast<double>(pb.scale) * 1.4426950408889634);
  p.n_qblk = (int)((pb.N_q + bm - 1) / bm);
  p.n_tiles = (int)(pb.B * pb.H * p.n_qblk);
  if (n_split > 1)
    p.n_split = n_split;
  else
    p.dv = dv;
  p.n_units = p.n_tiles * n_split;
  p.ws_o = ws.o;
  p.ws_lse = ws.lse;
  // Heads per schedule group: keep the K/V of a group within ~48 MB of L2
  // (24 MB under a causal mask: the longest-first order spreads the running
  // CTAs over more groups at once; measured +2 % on B4 H32 N8192 d128)
  // (K/V of every head within 64 MB: one group, so that the causal
  // longest-first order is global)
  const long long kv_bytes = pb.N_k * (pb.d + dv) * (fp32 ? 4 : 2);
  const long long budget = pb.is_causal ? (24ll << 20) : (48ll << 20);
  long long g = budget / (kv_bytes > 0 ? kv_bytes : 1);
  if (g < 1) g = 1;
  if (g > pb.B * pb.H || pb.B * kv_heads(pb) * kv_bytes <= (64ll << 20)) g = pb.B * pb.H;
  p.head_group = (int)g;
  p.kv_group = (int)(pb.H / kv_heads(pb));
  p.O = pb.O.ptr;
  for (int i = 0; i < 3; ++i) {
    p.o_stride[i] = pb.O.stride[i];
    p.lse_stride[i] = pb.LSE ? pb.lse_stride[i] : 0;
  }
  p.LSE = pb.LSE;
  p.err = ds.err;
  p.timeout_ns = g_timeout_ns.load();
  p.debug_flags = g_debug_flags.load();
  L.grid = p.n_units < ds.sm_count ? p.n_units : ds.sm_count;
  L.device = ds.device;
  L.stream = stream;
  cudaError_t e;
  if (vt) {
    VtParams v{};
    v.V = static_cast<const float*>(pb.V.ptr);
    v.s0 = pb.V.stride[0];
    v.s1 = pb.V.stride[1];
    v.s2 = pb.V.stride[2];
    v.Vt = vt;
    v.H_kv = (int)kv_heads(pb);
    v.N_k = (int)pb.N_k;
    v.dv = dv;
    v.ldk = (int)vt_ldk(pb.N_k);
    v.n_kblk = (int)((pb.N_k + kVtKeys - 1) / kVtKeys);
    fa_vt_kernel<<<(unsigned)(pb.B * kv_heads(pb) * v.n_kblk), 256, 0, stream>>>(v);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("V^T kernel launch", e));
    L.after_vt = true;
    e = d == 128 ? launch_tc_wide_fp32_d128_vt(L) : launch_tc_wide_fp32_d64_vt(L);
  } else if (fp32 && n_split > 1) {
    e = d == 128 ? launch_tc_wide_fp32_d128_split(L) : launch_tc_wide_fp32_d64_split(L);
  } else if (fp32) {
    e = d == 128 ? launch_tc_wide_fp32_d128(L) : launch_tc_wide_fp32_d64(L);
  } else if (wide) {
    e = launch_tc_wide_bf16_d256(L);
  } else if (n_split > 1) {
    e = d == 128 ? launch_tc_bf16_d128_split(L) : launch_tc_bf16_d64_split(L);
  } else {
    e = d == 128 ? launch_tc_bf16_d128(L) : (stages == 3 ? launch_tc_bf16_d64(L) : launch_tc_bf16_d64_causal(L));
  }
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("tensor-core kernel launch", e));
  if (n_split > 1) {
    CombineParams c{};
    c.B = (int)pb.B;
    c.H = (int)pb.H;
    c.N_q = (int)pb.N_q;
    c.N_k = (int)pb.N_k;
    c.causal = pb.is_causal != 0;
    c.causal_off = pb.is_causal == 2 ? (int)(pb.N_k - pb.N_q) : 0;
    c.n_split = n_split;
    c.bn = bn;
    c.bm = bm;
    c.rows = pb.B * pb.H * pb.N_q;
    c.ws_o = ws.o;
    c.ws_lse = ws.lse;
    c.O = pb.O.ptr;
    for (int i = 0; i < 3; ++i) {
      c.o_stride[i] = pb.O.stride[i];
      c.lse_stride[i] = pb.LSE ? pb.lse_stride[i] : 0;
    }
    c.LSE = pb.LSE;
    const unsigned blocks = (unsigned)((c.rows + 7) / 8);
    if (fp32)
      d == 128 ? fa_combine_kernel<float, 128><<<blocks, 256, 0, stream>>>(c)
               : fa_combine_kernel<float, 64><<<blocks, 256, 0, stream>>>(c);
    else
      d == 128 ? fa_combine_kernel<__nv_bfloat16, 128><<<blocks, 256, 0, stream>>>(c)
               : fa_combine_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, stream>>>(c);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("combine kernel launch", e));
  }
  return FA_OK;
}

// Split count for a problem (1 = do not split).  Work units run in waves of
// one per SM; a tile of n key tiles costs about n + 2 key-tile times (the 2
// covers its prologue and epilogue), so s splits take
//     ceil(tiles * s / SMs) * (n / s + 2)
// key-tile times.  A split is taken only if that is at least 10 % below the
// unsplit time and every split still covers >= 1024 keys (the partial-result
// round trip and the merge launch are not worth it for less).  Causal
// problems are balanced by their longest-first order, and the fp32 (tf32)
// path is not split automatically: on the measured fp32 shapes splitting was
// slower.  Callers can still ask for a split explicitly.
int choose_split(bool fp32, long long B, long long H, long long N_q, long long N_k, long long d, int causal,
                 int sm_count) {
  if (fp32 || causal || (d != 64 && d != 128) || sm_count <= 0) return 1;
  const int stages = tc_stages(fp32, (int)d, false, true);
  const long long bn = tc_key_tile(stages);
  const long long bm = tc_tile_rows(stages);
  const long long tiles = B * H * ((N_q + bm - 1) / bm);
  const long long n_kv = (N_k + bn - 1) / bn;
  auto cost = [&](long long s) {
    const long long waves = (tiles * s + sm_count - 1) / sm_count;
    return static_cast<double>(waves) * (static_cast<double>(n_kv) / s + 2.0);
  };
  const double base = cost(1);
  int best = 1;
  double best_cost = base;
  for (int s = 2; s <= 4; ++s) {
    if (N_k / s < 1024) break;
    const double c = cost(s);
    if (c < best_cost) {
      best_cost = c;
      best = s;
    }
  }
  return best_cost <= 0.9 * base ? best : 1;
}

bool row_aligned16(const fa_tensor_t& t, long long E) {
  if (reinterpret_cast<uintptr_t>(t.ptr) % 16 != 0) return false;
  for (int i = 0; i < 3; ++i)
    if ((t.stride[i] * E) % 16 != 0) return false;
  return true;
}

// fp32: warp-level tf32 tiles with a three-term split (fa_small_mma.cuh), one
// warp per work item, 4 per CTA; bf16: the CUDA-core kernel (fa_small.cuh),
// one CTA per work item.
template <typename T, int D>
cudaError_t launch_small_typed(const SmallParams& P, DevState& ds, cudaStream_t stream) {
  constexpr bool kMma = sizeof(T) == 4;
  constexpr int smem = kMma ? small_mma_smem_bytes<D>() : small_smem_bytes<T, D>();
  {  // once per device, so that captured launches make no attribute call
    std::lock_guard<std::mutex> lk(g_mu);
    bool& ready = ds.small_attr[sizeof(T) == 4 ? 1 : 0][D == 16 ? 0 : 1];
    if (!ready) {
      cudaError_t e;
      if constexpr (kMma)
        e = cudaFuncSetAttribute(fa_small_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      else
        e = cudaFuncSetAttribute(fa_small_fwd_kernel<T, D, kSmallSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
      if (e != cudaSuccess) return e;
      ready = true;
    }
  }
  if constexpr (kMma)
    fa_small_mma_kernel<D><<<(unsigned)((P.n_items + 1) / 2), 128, smem, stream>>>(P);
  else
    fa_small_fwd_kernel<T, D, kSmallSplit><<<(unsigned)P.n_items, 32 * kSmallSplit, smem, stream>>>(P);
  return cudaGetLastError();
}

// One launch for up to kSmallMaxGroup problems of the same dtype and head dim.
fa_status_t launch_small(fa_dtype_t dtype, int d, const std::vector<const fa_problem_t*>& probs,
                         DevState& ds, cudaStream_t stream) {
  const long long E = dtype == FA_FP32 ? 4 : 2;
  SmallParams P{};
  P.n_problems = (int)probs.size();
  long long items = 0;
  for (size_t i = 0; i < probs.size(); ++i) {
    const fa_problem_t& pb = *probs[i];
    SmallProblem& s = P.prob[i];
    s.Q = pb.Q.ptr;
    s.K = pb.K.ptr;
    s.V = pb.V.ptr;
    s.O = pb.O.ptr;
    s.LSE = pb.LSE;
    for (int k = 0; k < 3; ++k) {
      s.qs[k] = pb.Q.stride[k];
      s.ks[k] = pb.K.stride[k];
      s.vs[k] = pb.V.stride[k];
      s.os[k] = pb.O.stride[k];
      s.ls[k] = pb.LSE ? pb.lse_stride[k] : 0;
    }
    s.B = (int)pb.B;
    s.H = (int)pb.H;
    s.kv_group = (int)(pb.H / kv_heads(pb));
    s.N_q = (int)pb.N_q;
    s.N_k = (int)pb.N_k;
    s.causal = pb.is_causal != 0;
    s.causal_off = pb.is_causal == 2 ? (int)(pb.N_k - pb.N_q) : 0;
    s.scale_log2 = static_cast<float>(static_cast<double>(pb.scale) * 1.4426950408889634);
    s.n_qblk = (int)((pb.N_q + 31) / 32);
    s.vec_ok = row_aligned16(pb.Q, E) && row_aligned16(pb.K, E) && row_aligned16(pb.V, E) &&
               row_aligned16(pb.O, E);
    s.item_begin = items;
    items += pb.B * pb.H * s.n_qblk;
  }
  P.n_items = items;
  if (items >= (1ll << 31)) return fail(FA_ERR_UNSUPPORTED, "too many query blocks in one launch");
  cudaError_t e;
  if (dtype == FA_FP32)
    e = d == 16 ? launch_small_typed<float, 16>(P, ds, stream) : launch_small_typed<float, 32>(P, ds, stream);
  else
    e = d == 16 ? launch_small_typed<__nv_bfloat16, 16>(P, ds, stream)
                : launch_small_typed<__nv_bfloat16, 32>(P, ds, stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("small-head kernel launch", e));
  return FA_OK;
}

fa_status_t run_problems(fa_dtype_t dtype, int n, const fa_problem_t* problems, void* stream_ptr) {
  if (n < 0 || (n > 0 && !problems)) return fail(FA_ERR_INVALID_ARG, "bad problem list");
  std::vector<Path> paths(n);
  for (int i = 0; i < n; ++i) {
    fa_status_t st = validate(dtype, problems[i], i, &paths[i]);
    if (st != FA_OK) return st;
  }
  if (n == 0) return FA_OK;
  DevState* ds = nullptr;
  fa_status_t st = device_state(&ds);
  if (st != FA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  for (int d : {16, 32}) {
    std::vector<const fa_problem_t*> group;
    for (int i = 0; i < n; ++i) {
      if (paths[i] != Path::kSmall || problems[i].d != d) continue;
      group.push_back(&problems[i]);
      if ((int)group.size() == kSmallMaxGroup) {
        if ((st = launch_small(dtype, d, group, *ds, stream)) != FA_OK) return st;
        group.clear();
      }
    }
    if (!group.empty() && (st = launch_small(dtype, d, group, *ds, stream)) != FA_OK) return st;
  }
  for (int i = 0; i < n; ++i)
    if (paths[i] == Path::kTensorCore && (st = launch_tensor_core(dtype, problems[i], *ds, stream)) != FA_OK)
      return st;
  return FA_OK;
}

// The backward's fp32 dQ accumulator [BH][N_qp][D] as a 3-D tensor map for
// TMA reductions: boxes of 32 head dims x 64 query rows, unswizzled (D = 128),
// or 32 head dims x 32 query rows, 128-byte swizzle (D = 64).
fa_status_t make_dq_map(CUtensorMap* map, float* acc, long long BH, long long N_qp, long long D) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N_qp, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(D * 4), (cuuint64_t)(N_qp * D * 4)};
  cuuint32_t box[3] = {32, D == 128 ? 64u : 32u, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, acc, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, D == 128 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the dQ accumulator (CUresult " +
                                        std::to_string((int)r) + ")");
  return FA_OK;
}

// Backward workspace (caller-owned): fp32 dQ accumulator [B*H][N_qp][d], then
// -LSE * log2(e) and delta, [B*H][N_qp] each; every part 256-byte aligned.
// N_qp = N_q rounded up to the 128-row query tile.
struct BwdWs {
  float* dq_acc = nullptr;
  float* nlse2 = nullptr;
  float* delta = nullptr;
};
size_t bwd_part(size_t bytes) { return (bytes + 255) & ~size_t(255); }
size_t bwd_ws_bytes(long long B, long long H, long long N_q, long long d) {
  const size_t rows = static_cast<size_t>(B) * H * ((N_q + 127) / 128 * 128);
  return bwd_part(rows * d * 4) + 2 * bwd_part(rows * 4);
}
BwdWs bwd_ws_layout(void* ws, long long B, long long H, long long N_q, long long d) {
  const size_t rows = static_cast<size_t>(B) * H * ((N_q + 127) / 128 * 128);
  BwdWs w;
  char* c = static_cast<char*>(ws);
  w.dq_acc = reinterpret_cast<float*>(c);
  w.nlse2 = reinterpret_cast<float*>(c + bwd_part(rows * d * 4));
  w.delta = reinterpret_cast<float*>(c + bwd_part(rows * d * 4) + bwd_part(rows * 4));
  return w;
}

// A bf16 [B, H, N, d] view the backward reads or writes row-wise: non-null,
// unit inner stride, non-negative strides, 16-byte aligned base and strides.
fa_status_t check_bwd_tensor(const fa_tensor_t* t, const char* name) {
  if (!t || !tensor_ok(*t)) return fail(FA_ERR_INVALID_ARG, std::string(name) + " needs a non-null pointer and stride[3] == 1");
  if (reinterpret_cast<uintptr_t>(t->ptr) % 16 != 0)
    return fail(FA_ERR_UNSUPPORTED, std::string(name) + " must be 16-byte aligned");
  for (int i = 0; i < 3; ++i) {
    if (t->stride[i] < 0) return fail(FA_ERR_UNSUPPORTED, std::string(name) + ": negative strides are not supported");
    if ((t->stride[i] * 2) % 16 != 0)
      return fail(FA_ERR_UNSUPPORTED, std::string(name) + ": strides must be multiples of 16 bytes");
  }
  return FA_OK;
}

}  // namespace

namespace fa {
fa_status_t report_error(fa_status_t st, const std::string& msg) { return fail(st, msg); }
}  // namespace fa

extern "C" {

fa_status_t fa_fwd(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                   const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale, int is_causal,
                   const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3], void* stream) {
  return fa_fwd_gqa(dtype, B, H, H, N_q, N_k, d, Q, K, V, scale, is_causal, O, LSE, lse_stride, stream);
}

fa_status_t fa_fwd_gqa(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                       const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale, int is_causal,
                       const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3], void* stream) {
  if (!Q || !K || !V || !O) return fail(FA_ERR_INVALID_ARG, "Q, K, V and O must not be NULL");
  if (LSE && !lse_stride) return fail(FA_ERR_INVALID_ARG, "lse_stride must not be NULL when LSE is given");
  if (H_kv <= 0) return fail(FA_ERR_INVALID_ARG, "problem 0: H_kv must divide H");
  fa_problem_t pb{};
  pb.B = B;
  pb.H = H;
  pb.H_kv = H_kv;
  pb.N_q = N_q;
  pb.N_k = N_k;
  pb.d = d;
  pb.Q = *Q;
  pb.K = *K;
  pb.V = *V;
  pb.O = *O;
  pb.LSE = LSE;
  for (int i = 0; i < 3; ++i) pb.lse_stride[i] = LSE ? lse_stride[i] : 0;
  pb.scale = scale;
  pb.is_causal = is_causal;
  return run_problems(dtype, 1, &pb, stream);
}

fa_status_t fa_fwd_grouped(fa_dtype_t dtype, int n, const fa_problem_t* problems, void* stream) {
  return run_problems(dtype, n, problems, stream);
}

size_t fa_fwd_ws_bytes(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d) {
  if (dtype != FA_FP32 || B <= 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || N_q <= 0 || N_k <= 0 || d <= 0 ||
      d > kVtMaxDim || d == 16 || d == 32 || d % 4 != 0 || N_k >= (1ll << 31) || N_q >= (1ll << 31))
    return 0;
  fa_problem_t pb{};
  pb.B = B;
  pb.H = H;
  pb.H_kv = H_kv;
  pb.N_q = N_q;
  pb.N_k = N_k;
  pb.d = d;
  if (!wants_vt(dtype, pb, Path::kTensorCore)) return 0;
  return vt_ws_bytes(pb);
}

fa_status_t fa_fwd_ws(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                      const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale, int is_causal,
                      const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3], void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !O) return fail(FA_ERR_INVALID_ARG, "Q, K, V and O must not be NULL");
  if (LSE && !lse_stride) return fail(FA_ERR_INVALID_ARG, "lse_stride must not be NULL when LSE is given");
  if (H_kv <= 0) return fail(FA_ERR_INVALID_ARG, "problem 0: H_kv must divide H");
  fa_problem_t pb{};
  pb.B = B;
  pb.H = H;
  pb.H_kv = H_kv;
  pb.N_q = N_q;
  pb.N_k = N_k;
  pb.d = d;
  pb.Q = *Q;
  pb.K = *K;
  pb.V = *V;
  pb.O = *O;
  pb.LSE = LSE;
  for (int i = 0; i < 3; ++i) pb.lse_stride[i] = LSE ? lse_stride[i] : 0;
  pb.scale = scale;
  pb.is_causal = is_causal;
  Path path;
  fa_status_t st = validate(dtype, pb, 0, &path);
  if (st != FA_OK) return st;
  if (!wants_vt(dtype, pb, path)) return run_problems(dtype, 1, &pb, stream);  // no workspace needed
  if (B * H_kv * ((N_k + kVtKeys - 1) / kVtKeys) >= (1ll << 31)) return fail(FA_ERR_UNSUPPORTED, "too many V^T blocks");
  if (!workspace) return fail(FA_ERR_INVALID_ARG, "this problem needs a workspace (fa_fwd_ws_bytes > 0)");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(FA_ERR_INVALID_ARG, "the workspace must be 256-byte aligned");
  const size_t need = vt_ws_bytes(pb);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace too small: " + std::to_string(workspace_bytes) + " < " +
                                        std::to_string(need) + " bytes");
  DevState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  return launch_tensor_core(dtype, pb, *ds, static_cast<cudaStream_t>(stream), 1, SplitWs{},
                            static_cast<float*>(workspace));
}

size_t fa_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t N_q, int64_t d, int n_split) {
  if (B <= 0 || H <= 0 || N_q <= 0 || d <= 0 || n_split <= 1 || n_split > kMaxSplit) return 0;
  return split_ws_bytes(B, H, N_q, d, n_split);
}

int fa_fwd_splitkv_choose(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                          int is_causal) {
  if (B <= 0 || H <= 0 || N_q <= 0 || N_k <= 0) return 1;
  DevState* ds = nullptr;
  if (device_state(&ds) != FA_OK) return 1;
  return choose_split(dtype == FA_FP32, B, H, N_q, N_k, d, is_causal, ds->sm_count);
}

fa_status_t fa_fwd_splitkv(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                           const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                           int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                           int n_split, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_split < 1 || n_split > kMaxSplit)
    return fail(FA_ERR_INVALID_ARG, "n_split must be in [1, " + std::to_string(kMaxSplit) + "]");
  if (n_split == 1)
    return fa_fwd(dtype, B, H, N_q, N_k, d, Q, K, V, scale, is_causal, O, LSE, lse_stride, stream);
  if (!Q || !K || !V || !O) return fail(FA_ERR_INVALID_ARG, "Q, K, V and O must not be NULL");
  if (LSE && !lse_stride) return fail(FA_ERR_INVALID_ARG, "lse_stride must not be NULL when LSE is given");
  fa_problem_t pb{};
  pb.B = B;
  pb.H = H;
  pb.N_q = N_q;
  pb.N_k = N_k;
  pb.d = d;
  pb.Q = *Q;
  pb.K = *K;
  pb.V = *V;
  pb.O = *O;
  pb.LSE = LSE;
  for (int i = 0; i < 3; ++i) pb.lse_stride[i] = LSE ? lse_stride[i] : 0;
  pb.scale = scale;
  pb.is_causal = is_causal;
  Path path;
  fa_status_t st = validate(dtype, pb, 0, &path);
  if (st != FA_OK) return st;
  if (path != Path::kTensorCore || (d != 64 && d != 128))
    return fail(FA_ERR_UNSUPPORTED, "split-KV needs the tensor-core path with d = 64 or 128");
  if (B * H * ((N_q + 127) / 128) * n_split >= (1ll << 31))
    return fail(FA_ERR_UNSUPPORTED, "too many split-KV work units");
  if (!workspace) return fail(FA_ERR_INVALID_ARG, "split-KV needs a workspace");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(FA_ERR_INVALID_ARG, "the split-KV workspace must be 256-byte aligned");
  const size_t need = split_ws_bytes(B, H, N_q, d, n_split);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "split-KV workspace too small: " + std::to_string(workspace_bytes) + " < " +
                                        std::to_string(need) + " bytes");
  DevState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  return launch_tensor_core(dtype, pb, *ds, static_cast<cudaStream_t>(stream), n_split,
                            split_ws_layout(workspace, B, H, N_q, d, n_split));
}

size_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N_q, int64_t d) {
  if (B <= 0 || H <= 0 || N_q <= 0 || d <= 0 || d > 128 || N_q >= (1ll << 31)) return 0;
  return bwd_ws_bytes(B, H, N_q, tc_tile_dim(d, d));  // the accumulator has the tile's columns
}

fa_status_t fa_bwd(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k, int64_t d,
                   const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, const fa_tensor_t* O,
                   const fa_tensor_t* dO, const float* LSE, const int64_t lse_stride[3], float scale, int is_causal,
                   const fa_tensor_t* dQ, const fa_tensor_t* dK, const fa_tensor_t* dV, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return fa_bwd_gqa(dtype, B, H, H, N_q, N_k, d, Q, K, V, O, dO, LSE, lse_stride, scale, is_causal, dQ, dK, dV,
                    workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_gqa(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                       const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, const fa_tensor_t* O,
                       const fa_tensor_t* dO, const float* LSE, const int64_t lse_stride[3], float scale,
                       int is_causal, const fa_tensor_t* dQ, const fa_tensor_t* dK, const fa_tensor_t* dV,
                       void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_dv(dtype, B, H, H_kv, N_q, N_k, d, d, Q, K, V, O, dO, LSE, lse_stride, scale, is_causal, dQ, dK, dV,
                   workspace, workspace_bytes, stream);
}

fa_status_t fa_bwd_dv(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t N_q, int64_t N_k, int64_t d,
                      int64_t d_v, const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V,
                      const fa_tensor_t* O, const fa_tensor_t* dO, const float* LSE, const int64_t lse_stride[3],
                      float scale, int is_causal, const fa_tensor_t* dQ, const fa_tensor_t* dK,
                      const fa_tensor_t* dV, void* workspace, size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !O) return fail(FA_ERR_INVALID_ARG, "Q, K, V and O must not be NULL");
  if (H_kv <= 0) return fail(FA_ERR_INVALID_ARG, "H_kv must divide H");
  if (!LSE || !lse_stride) return fail(FA_ERR_INVALID_ARG, "the backward needs the forward's LSE and its strides");
  fa_problem_t pb{};
  pb.B = B;
  pb.H = H;
  pb.N_q = N_q;
  pb.N_k = N_k;
  pb.d = d;
  pb.Dv = d_v;
  pb.Q = *Q;
  pb.K = *K;
  pb.V = *V;
  pb.O = *O;
  pb.LSE = const_cast<float*>(LSE);
  for (int i = 0; i < 3; ++i) pb.lse_stride[i] = lse_stride[i];
  pb.scale = scale;
  pb.is_causal = is_causal;
  pb.H_kv = H_kv;
  Path path;
  fa_status_t st = validate(dtype, pb, 0, &path);
  if (st != FA_OK) return st;
  if (dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "the backward supports bf16 inputs only");
  if (d_v <= 0 || d > 128 || d_v > 128 || d % 8 != 0 || d_v % 8 != 0)
    return fail(FA_ERR_UNSUPPORTED, "the backward supports head dims d, d_v that are multiples of 8 up to 128");
  // the kernel's tile width: 64 or 128 columns; the columns of Q, K (past d) and
  // of V, dO (past d_v) load as zeros, and only d / d_v columns are stored
  const long long D = tc_tile_dim(d, d_v);
  if ((st = check_bwd_tensor(dO, "dO")) != FA_OK || (st = check_bwd_tensor(dQ, "dQ")) != FA_OK ||
      (st = check_bwd_tensor(dK, "dK")) != FA_OK || (st = check_bwd_tensor(dV, "dV")) != FA_OK)
    return st;
  const long long bm = D == 128 ? 64 : 128;  // query rows per step of the backward kernel
  const long long n_kt = (N_k + 127) / 128, n_qt = (N_q + bm - 1) / bm;
  if (B * H_kv * n_kt >= (1ll << 31) || B * H * n_qt * 128 >= (1ll << 40) || (H / H_kv) * n_qt >= (1ll << 31))
    return fail(FA_ERR_UNSUPPORTED, "too many backward work units");
  if (!workspace) return fail(FA_ERR_INVALID_ARG, "the backward needs a workspace");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(FA_ERR_INVALID_ARG, "the backward workspace must be 256-byte aligned");
  const size_t need = bwd_ws_bytes(B, H, N_q, D);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "backward workspace too small: " + std::to_string(workspace_bytes) + " < " +
                                        std::to_string(need) + " bytes");
  DevState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  const BwdWs ws = bwd_ws_layout(workspace, B, H, N_q, D);
  BwdLaunch L{};
  if ((st = make_map(&L.tmQ, *Q, false, B, H, N_q, (int)d, (int)bm, "Q")) != FA_OK) return st;
  if ((st = make_map(&L.tmdO, *dO, false, B, H, N_q, (int)d_v, (int)bm, "dO")) != FA_OK) return st;
  if ((st = make_map(&L.tmK, *K, false, B, H_kv, N_k, (int)d, 128, "K")) != FA_OK) return st;
  if ((st = make_map(&L.tmV, *V, false, B, H_kv, N_k, (int)d_v, 128, "V")) != FA_OK) return st;
  const int N_qp = (int)((N_q + 127) / 128 * 128);  // workspace row pitch
  if ((st = make_dq_map(&L.tmDq, ws.dq_acc, B * H, N_qp, D)) != FA_OK) return st;
  BwdParams& p = L.p;
  p.B = (int)B;
  p.H = (int)H;
  p.N_q = (int)N_q;
  p.N_k = (int)N_k;
  p.causal = is_causal != 0;
  p.causal_off = is_causal == 2 ? (int)(N_k - N_q) : 0;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.n_qt = (int)n_qt;
  p.n_kt = (int)n_kt;
  p.N_qp = N_qp;
  p.H_kv = (int)H_kv;
  p.kv_group = (int)(H / H_kv);
  p.n_units = (int)(B * H_kv * n_kt);
  {  // K/V heads per schedule group: their query heads' fp32 dQ rows, Q and dO within ~48 MB of L2
    const long long per_head = (N_qp * D * 4 + N_q * (d + d_v) * 2) * (H / H_kv);
    long long g = (48ll << 20) / (per_head > 0 ? per_head : 1);
    if (g < 1) g = 1;
    if (g > B * H_kv) g = B * H_kv;
    p.head_group = (int)g;
  }
  p.nlse2 = ws.nlse2;
  p.delta = ws.delta;
  p.dq_acc = ws.dq_acc;
  p.dK = dK->ptr;
  p.dV = dV->ptr;
  for (int i = 0; i < 3; ++i) {
    p.dk_stride[i] = dK->stride[i];
    p.dv_stride[i] = dV->stride[i];
  }
  p.err = ds->err;
  p.timeout_ns = g_timeout_ns.load();
  p.debug_flags = g_debug_flags.load();
  p.d_qk = (int)d;
  p.d_v = (int)d_v;
  BwdPreParams& pre = L.pre;
  pre.B = (int)B;
  pre.H = (int)H;
  pre.N_q = (int)N_q;
  pre.N_qp = N_qp;
  pre.O = O->ptr;
  pre.dO = dO->ptr;
  pre.LSE = LSE;
  for (int i = 0; i < 3; ++i) {
    pre.o_stride[i] = O->stride[i];
    pre.do_stride[i] = dO->stride[i];
    pre.lse_stride[i] = lse_stride[i];
  }
  pre.nlse2 = ws.nlse2;
  pre.delta = ws.delta;
  pre.dq_acc = ws.dq_acc;
  pre.d_v = (int)d_v;
  BwdPostParams& post = L.post;
  post.B = (int)B;
  post.H = (int)H;
  post.N_q = (int)N_q;
  post.N_qp = N_qp;
  post.scale = scale;
  post.dq_acc = ws.dq_acc;
  post.dQ = dQ->ptr;
  for (int i = 0; i < 3; ++i) post.dq_stride[i] = dQ->stride[i];
  post.d_qk = (int)d;
  L.d = (int)D;
  L.grid = p.n_units < ds->sm_count ? p.n_units : ds->sm_count;
  L.device = ds->device;
  L.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_bf16(L);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("backward launch", e));
  return FA_OK;
}

fa_status_t fa_fwd_varlen(fa_dtype_t dtype, int64_t B, int64_t H, int64_t H_kv, int64_t total_q, int64_t total_k,
                          int64_t max_len_q, int64_t d, int64_t d_v, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k,
                          const fa_tensor_t* Q, const fa_tensor_t* K, const fa_tensor_t* V, float scale,
                          int is_causal, const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                          void* stream) {
  if (!Q || !K || !V || !O) return fail(FA_ERR_INVALID_ARG, "Q, K, V and O must not be NULL");
  if (!cu_seqlens_q || !cu_seqlens_k) return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k are required");
  if (LSE && !lse_stride) return fail(FA_ERR_INVALID_ARG, "lse_stride must not be NULL when LSE is given");
  if (B <= 0 || max_len_q <= 0 || max_len_q > total_q || H_kv <= 0)
    return fail(FA_ERR_INVALID_ARG, "need B >= 1, H_kv >= 1 and 1 <= max_len_q <= total_q");
  // the packed tensors as [1, H, total, d] views: validate them like one problem
  fa_problem_t pb{};
  pb.B = 1;
  pb.H = H;
  pb.H_kv = H_kv;
  pb.N_q = total_q;
  pb.N_k = total_k;
  pb.d = d;
  pb.Dv = d_v;
  pb.Q = *Q;
  pb.K = *K;
  pb.V = *V;
  pb.O = *O;
  pb.LSE = LSE;
  for (int i = 0; i < 3; ++i) pb.lse_stride[i] = LSE ? lse_stride[i] : 0;
  pb.scale = scale;
  pb.is_causal = is_causal;
  Path path;
  fa_status_t st = validate(dtype, pb, 0, &path, /*tensor_core_only=*/true);
  if (st != FA_OK) return st;
  if (dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "packed variable-length batches take bf16");
  const int dv = static_cast<int>(v_dim(pb));
  const int D = tc_tile_dim(d, dv);
  if (D > 128) return fail(FA_ERR_UNSUPPORTED, "packed variable-length batches take head dims up to 128");
  const long long n_qblk = (max_len_q + 255) / 256;
  if (B * H * n_qblk >= (1ll << 31)) return fail(FA_ERR_UNSUPPORTED, "too many query tiles");
  DevState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  TcLaunch L;
  if ((st = make_map(&L.tmQ, pb.Q, false, 1, H, total_q, d, 128, "Q")) != FA_OK) return st;
  if ((st = make_map(&L.tmK, pb.K, false, 1, H_kv, total_k, d, 128, "K")) != FA_OK) return st;
  if ((st = make_map(&L.tmV, pb.V, false, 1, H_kv, total_k, dv, 128, "V")) != FA_OK) return st;
  if ((st = make_map(&L.tmO, pb.O, false, 1, H, total_q, dv, 32, "O")) != FA_OK) return st;
  TcParams& p = L.p;
  p.B = (int)B;
  p.H = (int)H;
  p.N_q = (int)total_q;
  p.N_k = (int)total_k;
  p.causal = is_causal == 0 ? kNoCausal : (is_causal == 2 ? kVarlenBottomRight : 0);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.n_qblk = (int)n_qblk;
  p.dv = dv;
  p.n_units = (int)(B * H * n_qblk);
  // this launch's work-unit counters: slots taken round robin, so that up to
  // kSchedSlots packed-batch launches may be in flight at once
  p.sched_slot = static_cast<int>(g_sched_next.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  // Heads per schedule group, as for the batched tiles: keep the K/V of a
  // group within ~48 MB of L2 (the longest query length stands in for the
  // key lengths, which only the device knows).
  const long long kv_bytes = max_len_q * (d + dv) * 2;
  long long hg = (48ll << 20) / (kv_bytes > 0 ? kv_bytes : 1);
  if (hg < 1) hg = 1;
  if (hg > B * H) hg = B * H;
  p.head_group = (int)hg;
  p.kv_group = (int)(H / H_kv);
  p.O = O->ptr;
  for (int i = 0; i < 3; ++i) {
    p.o_stride[i] = O->stride[i];
    p.lse_stride[i] = LSE ? lse_stride[i] : 0;
  }
  p.LSE = LSE;
  p.err = ds->err;
  p.timeout_ns = g_timeout_ns.load();
  p.debug_flags = g_debug_flags.load();
  L.grid = p.n_units < ds->sm_count ? p.n_units : ds->sm_count;
  L.device = ds->device;
  L.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = D == 128 ? launch_tc_bf16_d128_varlen(L) : launch_tc_bf16_d64_varlen(L);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("varlen kernel launch", e));
  return FA_OK;
}

fa_status_t fa_axial_block_fwd(int64_t B, int64_t H, int64_t W, int64_t D, int64_t heads, const float* x,
                               const fa_axial_weights_t* row, const fa_axial_weights_t* col, float* out,
                               void* stream) {
  if (!x || !out || !row || !col) return fail(FA_ERR_INVALID_ARG, "x, out and the weights must not be NULL");
  if (B <= 0 || H <= 0 || W <= 0) return fail(FA_ERR_INVALID_ARG, "B, H, W must be >= 1");
  if (D != kAxD || heads != kAxHeads)
    return fail(FA_ERR_UNSUPPORTED, "the fused axial block takes D = 64 with 4 heads");
  if (H > kAxMaxL || W > kAxMaxL) return fail(FA_ERR_UNSUPPORTED, "the fused axial block takes H, W <= 32");
  if (B * H * W * D >= (1ll << 40)) return fail(FA_ERR_UNSUPPORTED, "grid too large");
  const void* ptrs[] = {x, out, row->norm_w, row->norm_b, row->qkv_w, row->out_w, row->out_b,
                        col->norm_w, col->norm_b, col->qkv_w, col->out_w, col->out_b};
  for (const void* q : ptrs) {
    if (!q) return fail(FA_ERR_INVALID_ARG, "a weight pointer is NULL");
    if (reinterpret_cast<uintptr_t>(q) % 16 != 0)
      return fail(FA_ERR_UNSUPPORTED, "x, out and the weights must be 16-byte aligned");
  }
  DevState* ds = nullptr;
  fa_status_t st = device_state(&ds);
  if (st != FA_OK) return st;
  const int smem = static_cast<int>(sizeof(AxialSmem));
  {  // once per device (so that a captured launch makes no attribute call)
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ds->axial_attr) {
      cudaError_t e = cudaFuncSetAttribute(fa_axial_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("cudaFuncSetAttribute (axial block)", e));
      ds->axial_attr = true;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int pass = 0; pass < 2; ++pass) {
    const fa_axial_weights_t* wgt = pass == 0 ? row : col;
    AxialPassParams p{};
    p.x = pass == 0 ? x : out;  // the column pass reads the row pass's output
    p.out = out;
    p.outer_stride = H * W * D;
    if (pass == 0) {  // rows: sequence (b, h), tokens w
      p.n_seq = (int)(B * H);
      p.L = (int)W;
      p.seq_div = (int)H;
      p.inner_stride = W * D;
      p.tok_stride = D;
    } else {          // columns: sequence (b, w), tokens h
      p.n_seq = (int)(B * W);
      p.L = (int)H;
      p.seq_div = (int)W;
      p.inner_stride = D;
      p.tok_stride = W * D;
    }
    p.norm_w = wgt->norm_w;
    p.norm_b = wgt->norm_b;
    p.qkv_w = wgt->qkv_w;
    p.out_w = wgt->out_w;
    p.out_b = wgt->out_b;
    fa_axial_pass_kernel<<<p.n_seq, 256, smem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("axial block launch", e));
  }
  return FA_OK;
}

fa_status_t fa_check(void* stream_ptr) {
  DevState* ds = nullptr;
  fa_status_t st = device_state(&ds);
  if (st != FA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, cuda_msg("cudaStreamSynchronize", e));
  unsigned int word = 0;
  if ((e = cudaMemcpyAsync(&word, ds->err, sizeof(word), cudaMemcpyDeviceToHost, stream)) != cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess)
    return fail(FA_ERR_CUDA, cuda_msg("reading the device error word", e));
  if (word == 0) return FA_OK;
  if ((e = cudaMemsetAsync(ds->err, 0, sizeof(word), stream)) != cudaSuccess ||
      (e = cudaStreamSynchronize(stream)) != cudaSuccess)
    return fail(FA_ERR_CUDA, cuda_msg("clearing the device error word", e));
  char buf[128];
  std::snprintf(buf, sizeof(buf), "a bounded device wait expired (error word 0x%08x)", word);
  return fail(FA_ERR_TIMEOUT, buf);
}

const char* fa_status_string(fa_status_t status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported arguments";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* fa_last_error(void) { return t_last_error.c_str(); }

void fa_debug_set(uint64_t timeout_ns, int debug_flags) {
  g_timeout_ns.store(timeout_ns ? timeout_ns : 1000000000ull);
  g_debug_flags.store(debug_flags);
}

int fa_version(void) { return 105; }

}  // extern "C"
