// fa_launch.h -- internal interface between the C-ABI front end (fa_api.cu)
// and the translation units that instantiate the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "fa.h"
#include "fa_bwd.cuh"
#include "fa_tc.cuh"

namespace fa {

// Everything a tensor-core launch needs, prepared and validated on the host.
constexpr int kMaxDevices = 64;

struct TcLaunch {
  CUtensorMap tmQ, tmK, tmV;
  CUtensorMap tmO{};  // O, 32-row boxes (unsplit, not packed: TMA-store epilogue)
  TcParams p;
  int grid;
  int device;  // current device ordinal (per-device one-time setup)
  cudaStream_t stream;
  bool after_vt = false;  // launched behind fa_vt_kernel: programmatic dependent launch
};

// Kernel variants: (element type, head dim).  Each returns the CUDA error of
// the launch (cudaSuccess when it was queued).  Two-stage kernel (fa_tc.cuh),
// bf16, 256-row CTA tiles:
cudaError_t launch_tc_bf16_d128(const TcLaunch& L);
cudaError_t launch_tc_bf16_d64(const TcLaunch& L);         // three stages
cudaError_t launch_tc_bf16_d64_causal(const TcLaunch& L);  // two stages
// split-KV variants (L.p.n_split > 1, L.p.ws_o / ws_lse set)
cudaError_t launch_tc_bf16_d128_split(const TcLaunch& L);
cudaError_t launch_tc_bf16_d64_split(const TcLaunch& L);
// variable-length variants (bf16; L.p.cu_q / cu_k set, N_q / N_k = packed totals)
cudaError_t launch_tc_bf16_d128_varlen(const TcLaunch& L);
cudaError_t launch_tc_bf16_d64_varlen(const TcLaunch& L);
// single-stage kernel (fa_tc_wide.cuh): 128-row query blocks, 128-key tiles;
// bf16 head dims above 128 (up to 256) and every fp32 input (kind::tf32),
// the latter also split-KV
cudaError_t launch_tc_wide_bf16_d256(const TcLaunch& L);
cudaError_t launch_tc_wide_fp32_d128(const TcLaunch& L);
cudaError_t launch_tc_wide_fp32_d64(const TcLaunch& L);
cudaError_t launch_tc_wide_fp32_d128_split(const TcLaunch& L);
cudaError_t launch_tc_wide_fp32_d64_split(const TcLaunch& L);
// fp32 with V^T in global memory (tmV is then the map of V^T, fa_vt.cuh)
cudaError_t launch_tc_wide_fp32_d128_vt(const TcLaunch& L);
cudaError_t launch_tc_wide_fp32_d64_vt(const TcLaunch& L);
constexpr int kWideQueryTile = 128;
constexpr int kWideKeyTile = 128;

// Backward pass (fa_bwd.cu): preprocess, tensor-core kernel and dQ
// conversion on one stream.  bf16 only; d = 64 or 128.
struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmdO;
  CUtensorMap tmDq;  // the fp32 dQ accumulator [B*H][N_qp][d] (TMA reductions)
  BwdParams p;
  BwdPreParams pre;
  BwdPostParams post;
  int d;
  int grid;
  int device;
  cudaStream_t stream;
};
cudaError_t launch_bwd_bf16(const BwdLaunch& L);

// Records `msg` as the calling thread's fa_last_error() text and returns st
// (for entry points defined outside fa_api.cu).
fa_status_t report_error(fa_status_t st, const std::string& msg);

// Tile geometry shared with the instantiations in fa_tc_*.cu (the batched,
// not packed, two-stage kernel):
//  * query stages of a CTA tile: three for bf16 tiles of 64 columns when the
//    problem is not causal or is split (3 x (96 S + 64 O) tensor-memory
//    columns; measured +5..8 % on the d = 64 shapes, but -3 % causal, where
//    the larger diagonal block masks more work), else two;
//  * key-tile width: 96 keys with three stages, else 128;
//  * query rows of a CTA tile: 128 per stage;
//  * TMA box width: one 128-byte swizzle row, 64 bf16 or 32 fp32 values.
// (Packed batches keep two stages, 128-key tiles and 256-row virtual tiles.)
constexpr int tc_stages(bool fp32, int d, bool causal, bool split) {
  return (!fp32 && d <= 64 && (split || !causal)) ? 3 : 2;
}
constexpr int tc_key_tile(int stages) { return stages == 3 ? 96 : 128; }
constexpr int tc_tile_rows(int stages) { return 128 * stages; }
constexpr int tc_box_inner(bool fp32) { return fp32 ? 32 : 64; }

}  // namespace fa
