// fa_tc_fp32.cu -- fp32-input (tcgen05 kind::tf32) instantiations of the
// tensor-core forward kernel.  fp32 tiles are twice the bytes of bf16 ones and
// V also needs a transposed copy (tf32 B operands are K-major only), so key
// tiles are 32 (d = 128) or 64 (d = 64) wide to keep two 128-row Q tiles, the
// K/V ring and the V^T buffers in shared memory.
#include "fa_tc_inst.cuh"

namespace fa {

using CfgFp32D128 = TcCfg<float, 128, 32, 2>;
using CfgFp32D64 = TcCfg<float, 64, 64, 4>;
static_assert(tc_geometry_ok<CfgFp32D128, true>() && tc_geometry_ok<CfgFp32D64, true>(), "geometry");

cudaError_t launch_tc_fp32_d128(const TcLaunch& L) { return launch_tc<CfgFp32D128>(L); }
cudaError_t launch_tc_fp32_d64(const TcLaunch& L) { return launch_tc<CfgFp32D64>(L); }

}  // namespace fa
