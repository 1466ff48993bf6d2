// fa_tc_wide_fp32.cu -- fp32-input (tcgen05 kind::tf32) instantiations of the
// single-stage forward kernel (fa_tc_wide.cuh), unsplit and split-KV.
//  * d = 128: a 128-row fp32 tile of 128 columns has the byte geometry of a
//    bf16 tile of 256 (512-byte rows): Q 64 KB + a ring of 2 K/V slots of
//    64 KB, 128-key tiles; V^T is made in the ring slot (square tile);
//    S_0 | S_1 | O_0 | O_1 fill the 512 TMEM columns.
//  * d = 64: Q 32 KB + a ring of 4 slots of 32 KB + a 32 KB V^T buffer.
#include "fa_tc_inst.cuh"

namespace fa {

using CfgWideFp32D128 = TcWideCfg<float, 128, 128, 2>;
using CfgWideFp32D64 = TcWideCfg<float, 64, 128, 4>;
using CfgWideFp32D128Split = TcWideCfg<float, 128, 128, 2, true>;
using CfgWideFp32D64Split = TcWideCfg<float, 64, 128, 4, true>;
static_assert(CfgWideFp32D128::BN == kWideKeyTile && CfgWideFp32D128::BM == kWideQueryTile &&
                  CfgWideFp32D64::BN == kWideKeyTile && CfgWideFp32D64::BM == kWideQueryTile,
              "host tile geometry");
static_assert(CfgWideFp32D128::kPanelElems == tc_box_inner(true), "TMA box width");

cudaError_t launch_tc_wide_fp32_d128(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D128>(L); }
cudaError_t launch_tc_wide_fp32_d64(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D64>(L); }
cudaError_t launch_tc_wide_fp32_d128_split(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D128Split>(L); }
cudaError_t launch_tc_wide_fp32_d64_split(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D64Split>(L); }

}  // namespace fa
