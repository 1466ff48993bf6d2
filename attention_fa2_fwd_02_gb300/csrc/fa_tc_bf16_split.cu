// fa_tc_bf16_split.cu -- split-KV bf16 instantiations: the same tiles as
// fa_tc_bf16.cu, with work units that cover part of a tile's key range and
// write fp32 partial results to the caller's workspace.
#include <cuda_bf16.h>

#include "fa_tc_inst.cuh"

namespace fa {

using CfgBf16D128Split = TcCfg<__nv_bfloat16, 128, 128, 4, true>;
using CfgBf16D64Split = TcCfg<__nv_bfloat16, 64, 96, 10, true, false, 3>;
static_assert(tc_geometry_ok<CfgBf16D128Split, false>() && tc_geometry_ok<CfgBf16D64Split, false>(), "geometry");

cudaError_t launch_tc_bf16_d128_split(const TcLaunch& L) { return launch_tc<CfgBf16D128Split>(L); }
cudaError_t launch_tc_bf16_d64_split(const TcLaunch& L) { return launch_tc<CfgBf16D64Split>(L); }

}  // namespace fa
