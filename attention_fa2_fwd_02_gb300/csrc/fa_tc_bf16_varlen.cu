// fa_tc_bf16_varlen.cu -- variable-length (packed) bf16 instantiations: the
// same tiles as fa_tc_bf16.cu, over B packed sequences given by offsets.
#include <cuda_bf16.h>

#include "fa_tc_inst.cuh"

namespace fa {

using CfgBf16D128Varlen = TcCfg<__nv_bfloat16, 128, 128, 4, false, true>;
using CfgBf16D64Varlen = TcCfg<__nv_bfloat16, 64, 128, 6, false, true>;
// (packed batches: 128-key tiles and 256-row virtual tiles at both head dims,
// as fa_fwd_varlen sizes its tensor maps and tile grid)
static_assert(CfgBf16D128Varlen::BN == 128 && CfgBf16D64Varlen::BN == 128 && CfgBf16D128Varlen::kTileRows == 256 &&
                  CfgBf16D64Varlen::kTileRows == 256 && CfgBf16D64Varlen::kPanelElems == tc_box_inner(false),
              "geometry");

cudaError_t launch_tc_bf16_d128_varlen(const TcLaunch& L) { return launch_tc<CfgBf16D128Varlen>(L); }
cudaError_t launch_tc_bf16_d64_varlen(const TcLaunch& L) { return launch_tc<CfgBf16D64Varlen>(L); }

}  // namespace fa
