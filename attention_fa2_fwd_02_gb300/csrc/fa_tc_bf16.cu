// fa_tc_bf16.cu -- bf16 (tcgen05 kind::f16) instantiations of the tensor-core
// forward kernel: d = 128 with two query stages and a 4-deep ring of 128-key
// tiles; d = 64 with three query stages (three softmax warpgroups, each also
// storing its rows of O) and a 10-deep ring of 96-key tiles, or (causal) two
// stages and a 6-deep ring of 128-key tiles.
#include <cuda_bf16.h>

#include "fa_tc_inst.cuh"

namespace fa {

using CfgBf16D128 = TcCfg<__nv_bfloat16, 128, 128, 4>;
using CfgBf16D64 = TcCfg<__nv_bfloat16, 64, 96, 10, false, false, 3>;
using CfgBf16D64Causal = TcCfg<__nv_bfloat16, 64, 128, 6>;
static_assert(tc_geometry_ok<CfgBf16D128, false>() && tc_geometry_ok<CfgBf16D64, false>() &&
                  tc_geometry_ok<CfgBf16D64Causal, false>(),
              "geometry");

cudaError_t launch_tc_bf16_d128(const TcLaunch& L) { return launch_tc<CfgBf16D128>(L); }
cudaError_t launch_tc_bf16_d64(const TcLaunch& L) { return launch_tc<CfgBf16D64>(L); }
cudaError_t launch_tc_bf16_d64_causal(const TcLaunch& L) { return launch_tc<CfgBf16D64Causal>(L); }

}  // namespace fa
