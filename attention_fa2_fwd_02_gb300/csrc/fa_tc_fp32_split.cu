// fa_tc_fp32_split.cu -- split-KV fp32-input (tf32) instantiations: the same
// tiles as fa_tc_fp32.cu, with work units that cover part of a tile's key
// range and write fp32 partial results to the caller's workspace.
#include "fa_tc_inst.cuh"

namespace fa {

using CfgFp32D128Split = TcCfg<float, 128, 32, 2, true>;
using CfgFp32D64Split = TcCfg<float, 64, 64, 4, true>;
static_assert(tc_geometry_ok<CfgFp32D128Split, true>() && tc_geometry_ok<CfgFp32D64Split, true>(), "geometry");

cudaError_t launch_tc_fp32_d128_split(const TcLaunch& L) { return launch_tc<CfgFp32D128Split>(L); }
cudaError_t launch_tc_fp32_d64_split(const TcLaunch& L) { return launch_tc<CfgFp32D64Split>(L); }

}  // namespace fa
