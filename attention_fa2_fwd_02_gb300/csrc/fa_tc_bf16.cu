// fa_tc_bf16.cu -- bf16 (tcgen05 kind::f16) instantiations of the tensor-core
// forward kernel: d = 128 with a 4-deep ring of 128-key tiles, d = 64 with 6.
#include <cuda_bf16.h>

#include "fa_tc_inst.cuh"

namespace fa {

using CfgBf16D128 = TcCfg<__nv_bfloat16, 128, 128, 4>;
using CfgBf16D64 = TcCfg<__nv_bfloat16, 64, 128, 6>;
static_assert(tc_geometry_ok<CfgBf16D128, false>() && tc_geometry_ok<CfgBf16D64, false>(), "geometry");

cudaError_t launch_tc_bf16_d128(const TcLaunch& L) { return launch_tc<CfgBf16D128>(L); }
cudaError_t launch_tc_bf16_d64(const TcLaunch& L) { return launch_tc<CfgBf16D64>(L); }

}  // namespace fa
