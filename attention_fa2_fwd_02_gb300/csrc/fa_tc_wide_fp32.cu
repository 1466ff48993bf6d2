// fa_tc_wide_fp32.cu -- fp32-input (tcgen05 kind::tf32) instantiations of the
// single-stage forward kernel (fa_tc_wide.cuh), unsplit and split-KV.
// Q lives in tensor memory and its tiles travel through the K/V ring.
//  * d = 128: 128-row tiles of 512-byte rows (64 KB), a ring of 3 slots;
//    V^T is made in its ring slot (square tile); S_0 | S_1 | O | Q fill the
//    512 TMEM columns.
//  * d = 64: a ring of 5 slots of 32 KB and a 32 KB V^T buffer.
#include "fa_tc_inst.cuh"

namespace fa {

using CfgWideFp32D128 = TcWideCfg<float, 128, 128, 3>;
using CfgWideFp32D64 = TcWideCfg<float, 64, 128, 5>;
using CfgWideFp32D128Split = TcWideCfg<float, 128, 128, 3, true>;
using CfgWideFp32D64Split = TcWideCfg<float, 64, 128, 5, true>;
static_assert(CfgWideFp32D128::BN == kWideKeyTile && CfgWideFp32D128::BM == kWideQueryTile &&
                  CfgWideFp32D64::BN == kWideKeyTile && CfgWideFp32D64::BM == kWideQueryTile,
              "host tile geometry");
static_assert(CfgWideFp32D128::kPanelElems == tc_box_inner(true), "TMA box width");

cudaError_t launch_tc_wide_fp32_d128(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D128>(L); }
cudaError_t launch_tc_wide_fp32_d64(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D64>(L); }
cudaError_t launch_tc_wide_fp32_d128_split(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D128Split>(L); }
cudaError_t launch_tc_wide_fp32_d64_split(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D64Split>(L); }

}  // namespace fa
