// fa_axial_block.cuh -- the axial attention block fused per sequence (fp32).
//
// The module of the axial-attention transcript (its _attn_ref and forward):
// on x [B, H, W, D], a row pass over the W-long rows, then a column pass over
// the H-long columns of the updated grid; each pass is
//     x += out_proj(attention(qkv_proj(LayerNorm(x))))
// with LayerNorm (biased variance, eps 1e-5, affine), a bias-free QKV
// projection [3D, D], softmax(q k^T / sqrt(d)) v per head, and an output
// projection [D, D] with bias.  D = 64, 4 heads of 16, sequences of <= 32
// tokens: the shapes of the transcript's module.
//
// One CTA (256 threads) per sequence does the whole pass in shared memory:
// the weights (rows padded by one word, so that a warp's reads of one k
// across its output rows fall in different banks), the sequence, LayerNorm (a warp per token, shuffle
// reductions inside the warp), the QKV projection (each thread a 4 x 6
// register tile), the attention (a thread per (head, query)), the output
// projection with bias and the residual.  The column pass reads the row
// pass's output; both passes may run in place (a CTA reads its whole
// sequence before it writes any of it, and sequences are disjoint).
#pragma once

#include <cuda_runtime.h>

namespace fa {

constexpr int kAxD = 64, kAxHeads = 4, kAxHd = 16, kAxMaxL = 32;

struct AxialPassParams {
  const float* x;      // input grid [B, H, W, D]
  float* out;          // output grid [B, H, W, D] (may be x)
  int n_seq;           // sequences of this pass
  int L;               // tokens per sequence
  int seq_div;         // sequence s = (s / seq_div, s % seq_div) -> base offset below
  long long outer_stride, inner_stride;  // elements: base = (s / seq_div) * outer + (s % seq_div) * inner
  long long tok_stride;                  // elements between consecutive tokens
  const float* norm_w;
  const float* norm_b;
  const float* qkv_w;  // [3D, D]
  const float* out_w;  // [D, D]
  const float* out_b;  // [D]
};

constexpr int kAxQkvLd = 3 * kAxD + 4;  // padded row of the qkv buffer
constexpr int kAxWLd = kAxD + 1;        // padded weight row: a warp's reads of one k in 32 rows spread over the banks
struct AxialSmem {
  float wqkv[3 * kAxD][kAxWLd];   // qkv_w as given: [o][k]
  float wo[kAxD][kAxWLd];         // out_w as given: [o][k]
  float x[kAxMaxL][kAxD];
  float xn[kAxMaxL][kAxD];
  float qkv[kAxMaxL][kAxQkvLd];
  float ao[kAxMaxL][kAxD];
  float nw[kAxD], nb[kAxD], ob[kAxD];
};

__global__ void __launch_bounds__(256) fa_axial_pass_kernel(const __grid_constant__ AxialPassParams p) {
  extern __shared__ __align__(16) unsigned char ax_smem_raw[];
  AxialSmem& sm = *reinterpret_cast<AxialSmem*>(ax_smem_raw);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int s = blockIdx.x;
  const long long base = (s / p.seq_div) * p.outer_stride + (s % p.seq_div) * p.inner_stride;
  const int L = p.L;

  // weights in their [o][k] layout, rows padded to kAxWLd (consecutive
  // threads store consecutive words: no bank conflicts)
  for (int i = tid; i < 3 * kAxD * kAxD / 4; i += 256) {
    const float4 w = reinterpret_cast<const float4*>(p.qkv_w)[i];
    float* dst = &sm.wqkv[(4 * i) / kAxD][(4 * i) % kAxD];
    dst[0] = w.x;
    dst[1] = w.y;
    dst[2] = w.z;
    dst[3] = w.w;
  }
  for (int i = tid; i < kAxD * kAxD / 4; i += 256) {
    const float4 w = reinterpret_cast<const float4*>(p.out_w)[i];
    float* dst = &sm.wo[(4 * i) / kAxD][(4 * i) % kAxD];
    dst[0] = w.x;
    dst[1] = w.y;
    dst[2] = w.z;
    dst[3] = w.w;
  }
  if (tid < kAxD) {
    sm.nw[tid] = p.norm_w[tid];
    sm.nb[tid] = p.norm_b[tid];
    sm.ob[tid] = p.out_b[tid];
  }
  // the sequence (tokens past L are zero)
  for (int i = tid; i < kAxMaxL * kAxD / 4; i += 256) {
    const int t = (4 * i) / kAxD, c = (4 * i) % kAxD;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < L) v = *reinterpret_cast<const float4*>(p.x + base + t * p.tok_stride + c);
    *reinterpret_cast<float4*>(&sm.x[t][c]) = v;
  }
  __syncthreads();

  // LayerNorm: warp w takes tokens w, w + 8, ...; lane holds columns lane, lane + 32
  for (int t = warp; t < kAxMaxL; t += 8) {
    const float a = sm.x[t][lane], b = sm.x[t][lane + 32];
    float sum = a + b;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum * (1.f / kAxD);
    const float da = a - mean, db = b - mean;
    float sq = da * da + db * db;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    const float inv = rsqrtf(sq * (1.f / kAxD) + 1e-5f);
    const bool live = t < L;
    sm.xn[t][lane] = live ? da * inv * sm.nw[lane] + sm.nb[lane] : 0.f;
    sm.xn[t][lane + 32] = live ? db * inv * sm.nw[lane + 32] + sm.nb[lane + 32] : 0.f;
  }
  __syncthreads();

  // QKV projection: warp w -> tokens 4w .. 4w+3, lane -> outputs 6 lane .. 6 lane + 5
  {
    float acc[4][6] = {};
    const int t0 = 4 * warp, o0 = 6 * lane;
#pragma unroll 8
    for (int k = 0; k < kAxD; ++k) {
      float xv[4], wv[6];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = sm.xn[t0 + i][k];
#pragma unroll
      for (int j = 0; j < 6; ++j) wv[j] = sm.wqkv[o0 + j][k];  // banks (6 lane + j + k) mod 32: 2-way at most
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 6; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 6; ++j) sm.qkv[t0 + i][o0 + j] = acc[i][j];
  }
  __syncthreads();

  // attention: thread (head, query) for the first 128 threads
  if (tid < kAxHeads * kAxMaxL) {
    const int head = tid / kAxMaxL, q = tid % kAxMaxL;
    if (q < L) {
      const float scale = 0.25f;  // 1 / sqrt(16)
      float qv[kAxHd];
#pragma unroll
      for (int c = 0; c < kAxHd; ++c) qv[c] = sm.qkv[q][head * kAxHd + c] * scale;
      float sc[kAxMaxL];
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < kAxMaxL; ++j) {
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < kAxHd; ++c) dot = fmaf(qv[c], sm.qkv[j][kAxD + head * kAxHd + c], dot);
        sc[j] = j < L ? dot : -INFINITY;
        m = fmaxf(m, sc[j]);
      }
      float l = 0.f, o[kAxHd] = {};
#pragma unroll
      for (int j = 0; j < kAxMaxL; ++j) {
        const float pj = j < L ? __expf(sc[j] - m) : 0.f;
        l += pj;
#pragma unroll
        for (int c = 0; c < kAxHd; ++c) o[c] = fmaf(pj, sm.qkv[j][2 * kAxD + head * kAxHd + c], o[c]);
      }
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < kAxHd; ++c) sm.ao[q][head * kAxHd + c] = o[c] * inv;
    } else {
#pragma unroll
      for (int c = 0; c < kAxHd; ++c) sm.ao[q][head * kAxHd + c] = 0.f;
    }
  }
  __syncthreads();

  // output projection + bias + residual: warp w -> tokens 4w .. 4w+3, lane -> outputs 2 lane, 2 lane + 1
  {
    const int t0 = 4 * warp, o0 = 2 * lane;
    float acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i][0] = sm.x[t0 + i][o0] + sm.ob[o0];
      acc[i][1] = sm.x[t0 + i][o0 + 1] + sm.ob[o0 + 1];
    }
#pragma unroll 8
    for (int k = 0; k < kAxD; ++k) {
      const float w0 = sm.wo[o0][k], w1 = sm.wo[o0 + 1][k];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = sm.ao[t0 + i][k];
        acc[i][0] = fmaf(a, w0, acc[i][0]);
        acc[i][1] = fmaf(a, w1, acc[i][1]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (t0 + i < L)
        *reinterpret_cast<float2*>(p.out + base + (t0 + i) * p.tok_stride + o0) = make_float2(acc[i][0], acc[i][1]);
  }
}

}  // namespace fa
