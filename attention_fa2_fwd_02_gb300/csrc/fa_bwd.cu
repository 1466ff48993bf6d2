// fa_bwd.cu -- instantiations and launch of the backward pass (bf16, head dims
// 64 and 128): the preprocess, the tensor-core kernel and the dQ conversion,
// queued on one stream.
#include <cuda_bf16.h>

#include <atomic>

#include "fa_launch.h"

namespace fa {

template <int D>
static cudaError_t launch_bwd_d(const BwdLaunch& L) {
  using C = BwdCfg<D>;
  static std::atomic<bool> ready[kMaxDevices];
  if (L.device < 0 || L.device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!ready[L.device].load(std::memory_order_acquire)) {  // once per device (no attribute call when captured)
    cudaError_t e = cudaFuncSetAttribute(fa_bwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    ready[L.device].store(true, std::memory_order_release);
  }
  const long long pre_rows = static_cast<long long>(L.pre.B) * L.pre.H * L.pre.N_qp;
  fa_bwd_pre_kernel<__nv_bfloat16, D><<<(unsigned)((pre_rows + 7) / 8), 256, 0, L.stream>>>(L.pre);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_kernel<C><<<L.grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.tmdO, L.p, L.tmDq);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long post_rows = static_cast<long long>(L.post.B) * L.post.H * L.post.N_q;
  fa_bwd_post_kernel<__nv_bfloat16, D><<<(unsigned)((post_rows + 7) / 8), 256, 0, L.stream>>>(L.post);
  return cudaGetLastError();
}

cudaError_t launch_bwd_bf16(const BwdLaunch& L) { return L.d == 128 ? launch_bwd_d<128>(L) : launch_bwd_d<64>(L); }

}  // namespace fa
