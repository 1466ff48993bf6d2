// fa_tc_wide_fp32_vt.cu -- fp32-input (tcgen05 kind::tf32) instantiations of
// the single-stage forward kernel (fa_tc_wide.cuh) that read V^T, written to
// global memory by fa_vt_kernel (fa_vt.cuh), instead of transposing V tiles
// in shared memory.  Q stays in shared memory and O is double-buffered in
// tensor memory, as for bf16 d = 256 (whose tiles have the same bytes).
//  * d = 128: a ring of 2 slots of 64 KB next to the 64 KB Q tile;
//  * d = 64: a ring of 5 slots of 32 KB next to the 32 KB Q tile.
#include "fa_tc_inst.cuh"

namespace fa {

using CfgWideFp32D128Vt = TcWideCfg<float, 128, 128, 2, false, true>;
using CfgWideFp32D64Vt = TcWideCfg<float, 64, 128, 5, false, true>;
static_assert(CfgWideFp32D128Vt::BN == kWideKeyTile && CfgWideFp32D128Vt::BM == kWideQueryTile &&
                  CfgWideFp32D64Vt::BN == kWideKeyTile && CfgWideFp32D64Vt::BM == kWideQueryTile,
              "host tile geometry");
static_assert(CfgWideFp32D128Vt::kOBufs == 2 && CfgWideFp32D64Vt::kOBufs == 2, "double-buffered O");

cudaError_t launch_tc_wide_fp32_d128_vt(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D128Vt>(L); }
cudaError_t launch_tc_wide_fp32_d64_vt(const TcLaunch& L) { return launch_tc_wide<CfgWideFp32D64Vt>(L); }

}  // namespace fa
