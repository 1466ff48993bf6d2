// fa_tc_bf16.cu -- bf16 (tcgen05 kind::f16) instantiations of the tensor-core
// forward kernel: d = 128 with a 4-deep ring of 128-key tiles, d = 64 with 6.
#include <cuda_bf16.h>

#include <atomic>

#include "fa_launch.h"

namespace fa {

using CfgBf16D128 = TcCfg<__nv_bfloat16, 128, 128, 4>;
using CfgBf16D64 = TcCfg<__nv_bfloat16, 64, 128, 6>;
static_assert(CfgBf16D128::BN == tc_key_tile(false, 128) && CfgBf16D64::BN == tc_key_tile(false, 64), "geometry");
static_assert(CfgBf16D128::kPanelElems == tc_box_inner(false), "geometry");

// The shared-memory opt-in is set once per device (so that a launch captured
// into a CUDA graph makes no attribute call).
template <class C>
static cudaError_t launch(const TcLaunch& L) {
  static std::atomic<bool> ready[kMaxDevices];
  if (L.device < 0 || L.device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!ready[L.device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(fa_tc_fwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    ready[L.device].store(true, std::memory_order_release);
  }
  fa_tc_fwd_kernel<C><<<L.grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.p);
  return cudaGetLastError();
}

cudaError_t launch_tc_bf16_d128(const TcLaunch& L) { return launch<CfgBf16D128>(L); }
cudaError_t launch_tc_bf16_d64(const TcLaunch& L) { return launch<CfgBf16D64>(L); }

}  // namespace fa
