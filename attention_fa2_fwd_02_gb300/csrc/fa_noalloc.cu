// fa_noalloc.cu -- the split-KV forward for callers that cannot allocate
// device memory (fa_fwd_splitkv_noalloc in fa.h).
//
// The partial results of the split kernel go to one fixed scratch buffer per
// device: a static device array of this translation unit, so the CUDA runtime
// places it on a device when it loads this unit's module there (on first use,
// under lazy module loading).  Nothing here calls an allocator.  The source
// pages have no counterpart: this only changes where the scratch lives.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <string>

#include "fa.h"
#include "fa_combine.cuh"
#include "fa_launch.h"

namespace fa {

constexpr size_t kNoAllocScratchBytes = FA_SPLITKV_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size");

// The scratch itself (256-byte aligned, as fa_fwd_splitkv requires).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mu;
std::atomic<void*> g_scratch_ptr[kMaxDevices];  // device address per ordinal, once looked up

// Device address of the scratch on the current device.  The first call per
// device looks it up with that device current and caches it (for the life of
// the process: cudaDeviceReset while the library is loaded is not supported).
fa_status_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return report_error(FA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return report_error(FA_ERR_CUDA, "device ordinal out of range");
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p)
        return report_error(FA_ERR_CUDA, std::string("cudaGetSymbolAddress(no-alloc scratch): ") +
                                             cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status_t fa_fwd_splitkv_noalloc(fa_dtype_t dtype, int64_t B, int64_t H, int64_t N_q, int64_t N_k,
                                              int64_t d, const fa_tensor_t* Q, const fa_tensor_t* K,
                                              const fa_tensor_t* V, float scale, int is_causal,
                                              const fa_tensor_t* O, float* LSE, const int64_t lse_stride[3],
                                              int n_split, void* stream) {
  using namespace fa;
  // n_split = 1 (no scratch) and out-of-range n_split: fa_fwd_splitkv's own
  // handling, with no workspace
  if (n_split < 2 || n_split > kMaxSplit)
    return fa_fwd_splitkv(dtype, B, H, N_q, N_k, d, Q, K, V, scale, is_causal, O, LSE, lse_stride, n_split,
                          nullptr, 0, stream);
  // Size check before anything else, in floating point so that absurd sizes
  // cannot wrap around; non-positive sizes fall through to the argument
  // checks of fa_fwd_splitkv.
  if (B > 0 && H > 0 && N_q > 0 && d > 0) {
    const double need_est = static_cast<double>(n_split) * static_cast<double>(B) * static_cast<double>(H) *
                            static_cast<double>(N_q) * (4.0 * static_cast<double>(d) + 4.0);
    const bool huge = need_est >= 1e18;
    const size_t need = huge ? 0 : fa_fwd_splitkv_workspace_bytes(B, H, N_q, d, n_split);
    if (huge || need > kNoAllocScratchBytes)
      return report_error(FA_ERR_UNSUPPORTED,
                          "split-KV with n_split=" + std::to_string(n_split) + " needs " +
                              (huge ? std::string("more than 1e18") : std::to_string(need)) +
                              " bytes of scratch; the built-in no-alloc buffer holds " +
                              std::to_string(kNoAllocScratchBytes) +
                              " (use fewer splits, or fa_fwd_splitkv with a caller workspace)");
  }
  void* scratch = nullptr;
  fa_status_t st = scratch_on_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_fwd_splitkv(dtype, B, H, N_q, N_k, d, Q, K, V, scale, is_causal, O, LSE, lse_stride, n_split, scratch,
                        kNoAllocScratchBytes, stream);
}
