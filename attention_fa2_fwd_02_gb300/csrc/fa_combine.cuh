// fa_combine.cuh -- merge of split-KV partial results.
//
// With the key range of a query tile cut into splits, split s produces for
// every row its own normalised output O_s = sum_{j in s} e^{s_j - L_s} V_j and
// LSE L_s = log sum_{j in s} e^{s_j}.  The full result follows from the same
// identity the online softmax uses ("Extend Thunder with CUDA-Python",
// flash_attention_reference: rescale by the exponential of the difference of
// the log-sum-exps):
//     L = log sum_s e^{L_s},   O = sum_s e^{L_s - L} O_s.
// A split none of whose keys a row sees (causal) has O_s = 0, L_s = -inf and
// weight 0; a row that sees no key at all gets O = 0, L = -inf.  One warp per row; each lane owns D/32 consecutive columns.
#pragma once

#include "fa_ptx.cuh"

namespace fa {

constexpr int kMaxSplit = 8;

struct CombineParams {
  int B, H, N_q, N_k, causal, n_split, bn;  // bn: key-tile width used by the split kernel
  int bm;                                   // query rows of a tile of the split kernel
  int causal_off;                           // as TcParams::causal_off
  long long rows;                           // B * H * N_q
  const float* ws_o;                        // [n_split][rows][D]
  const float* ws_lse;                      // [n_split][rows]
  void* O;
  long long o_stride[3];
  float* LSE;
  long long lse_stride[3];
};

template <typename T, int D>
__global__ void __launch_bounds__(256) fa_combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr int PER = D / 32;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32;
  if (row >= p.rows) return;
  const int lane = threadIdx.x & 31;
  const int q = static_cast<int>(row % p.N_q);
  const long long bh = row / p.N_q;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  // splits that exist for this row's tile (same rule as the split kernel)
  const int q0 = (q / p.bm) * p.bm;
  int kv_end = p.N_k;
  if (p.causal) kv_end = min(kv_end, min(q0 + p.bm, p.N_q) + p.causal_off);
  const int n_tot = kv_end > 0 ? (kv_end + p.bn - 1) / p.bn : 0;
  const int s_eff = min(p.n_split, n_tot);

  float lse_s[kMaxSplit];
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s) {
    lse_s[s] = s < s_eff ? p.ws_lse[s * p.rows + row] : -INFINITY;
    m = fmaxf(m, lse_s[s]);
  }
  float l = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s)
    if (s < s_eff && m != -INFINITY) l += expf(lse_s[s] - m);
  // a row that sees no key in any split (bottom-right causal, N_q > N_k):
  // l = 0, so LSE = -inf and every weight below is 0
  const float lse = m == -INFINITY ? -INFINITY : m + logf(l);

  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s) {
    if (s >= s_eff) break;
    const float w = lse == -INFINITY ? 0.f : expf(lse_s[s] - lse);
    const float* src = p.ws_o + (s * p.rows + row) * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
    }
  }
  T* dst = reinterpret_cast<T*>(p.O) + b * p.o_stride[0] + h * p.o_stride[1] +
           static_cast<long long>(q) * p.o_stride[2] + lane * PER;
  if constexpr (sizeof(T) == 4) {
    if constexpr (PER == 4)
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else
      *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
  } else {
    if constexpr (PER == 4)
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
    else
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
  }
  if (lane == 0 && p.LSE)
    p.LSE[b * p.lse_stride[0] + h * p.lse_stride[1] + static_cast<long long>(q) * p.lse_stride[2]] = lse;
}

}  // namespace fa
