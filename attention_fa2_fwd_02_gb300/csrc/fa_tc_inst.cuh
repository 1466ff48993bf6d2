// fa_tc_inst.cuh -- launch wrapper shared by the translation units that
// instantiate the tensor-core kernel (one variant family per unit, so that
// they compile in parallel).
#pragma once

#include <atomic>

#include "fa_launch.h"
#include "fa_tc_wide.cuh"

namespace fa {

// The shared-memory opt-in is set once per device (so that a launch captured
// into a CUDA graph makes no attribute call).
template <class C>
static cudaError_t launch_tc(const TcLaunch& L) {
  static std::atomic<bool> ready[kMaxDevices];
  if (L.device < 0 || L.device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!ready[L.device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(fa_tc_fwd_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    ready[L.device].store(true, std::memory_order_release);
  }
  fa_tc_fwd_kernel<C><<<L.grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.tmO, L.p);
  return cudaGetLastError();
}

// The same for the single-stage kernel (fa_tc_wide.cuh).
template <class C>
static cudaError_t launch_tc_wide(const TcLaunch& L) {
  static std::atomic<bool> ready[kMaxDevices];
  if (L.device < 0 || L.device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!ready[L.device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(fa_tc_wide_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    ready[L.device].store(true, std::memory_order_release);
  }
  if (!L.after_vt) {
    fa_tc_wide_kernel<C><<<L.grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tmQ, L.tmK, L.tmV, L.tmO, L.p);
    return cudaGetLastError();
  }
  // behind the V^T pass: start early (barriers, tensor memory, Q and K
  // copies); the load warp waits for the pass before its first V^T copy
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(L.grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_tc_wide_kernel<C>, L.tmQ, L.tmK, L.tmV, L.tmO, L.p);
}

// Geometry of the instantiated configurations (the host side sizes its TMA
// boxes from tc_key_tile / tc_box_inner).
template <class C, bool FP32>
constexpr bool tc_geometry_ok() {
  return C::BN == tc_key_tile(C::NST) && C::kTileRows == tc_tile_rows(C::NST) &&
         C::kPanelElems == tc_box_inner(FP32);
}

}  // namespace fa
