// fa_tc_fp32.cu -- fp32-input (tcgen05 kind::tf32) instantiations of the
// tensor-core forward kernel.  fp32 tiles are twice the bytes of bf16 ones and
// V also needs a transposed copy (tf32 B operands are K-major only), so key
// tiles are 32 (d = 128) or 64 (d = 64) wide to keep two 128-row Q tiles, the
// K/V ring and the V^T buffers in shared memory.
#include <atomic>

#include "fa_launch.h"

namespace fa {

using CfgFp32D128 = TcCfg<float, 128, 32, 2>;
using CfgFp32D64 = TcCfg<float, 64, 64, 4>;
static_assert(CfgFp32D128::BN == tc_key_tile(true, 128) && CfgFp32D64::BN == tc_key_tile(true, 64), "geometry");
static_assert(CfgFp32D128::kPanelElems == tc_box_inner(true), "geometry");

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

cudaError_t launch_tc_fp32_d128(const TcLaunch& L) { return launch<CfgFp32D128>(L); }
cudaError_t launch_tc_fp32_d64(const TcLaunch& L) { return launch<CfgFp32D64>(L); }

}  // namespace fa
