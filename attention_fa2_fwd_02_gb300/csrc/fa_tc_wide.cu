// fa_tc_wide.cu -- the bf16 forward for head dims above 128 (up to 256): one
// 128-row query block per CTA tile, 128-key tiles, a ring of 2 K/V slots
// (Q 64 KB + 2 x 64 KB of shared memory; S_0 | S_1 | O fill the 512 TMEM
// columns).  Measured against 64-key tiles with 4 or 5 slots, the wider key
// tile is 15-20 % faster: the softmax's fixed cost per tile (waits, row max
// tree, hand-offs) is paid half as often, and two slots still cover the loads.
#include <cuda_bf16.h>

#include "fa_tc_inst.cuh"

namespace fa {

using CfgWideD256 = TcWideCfg<__nv_bfloat16, 256, 128, 2>;
static_assert(CfgWideD256::BN == kWideKeyTile && CfgWideD256::BM == kWideQueryTile, "host tile geometry");

cudaError_t launch_tc_wide_bf16_d256(const TcLaunch& L) { return launch_tc_wide<CfgWideD256>(L); }

}  // namespace fa
