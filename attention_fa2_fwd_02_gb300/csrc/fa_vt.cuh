// fa_vt.cuh -- V^T for the tf32 tensor-core path: one pass over V that writes
// it transposed, keys contiguous, into the caller's workspace.
//
// Why: P.V takes V as the B operand of a tf32 tcgen05.mma, and the tensor
// core takes tf32 operands only K-major, i.e. with the reduction index (the
// key) contiguous.  V [B, H_kv, N_k, Dv] has the head dims contiguous.  The
// attention kernel can transpose each V tile in shared memory (its warpgroup
// 1 does, when no workspace is given), but then every query tile that reads a
// V tile transposes it again, and the shared-memory traffic of that
// transpose, next to the tensor core's own operand reads, sets the pace of
// the kernel.  Written once to global memory instead, V^T costs one read and
// one write of V (an HBM-bound pass), and the attention kernel loads V^T
// tiles with TMA exactly like K tiles.
//
// Layout of V^T: [B * H_kv][Dv][ldk] fp32, element (b, h, c, n) =
// V[b, h, n, c]; ldk = N_k rounded up to 32 (128-byte rows, so that every
// warp's 32-key store is one aligned line).  Columns n >= N_k are never
// written: the tensor map's key extent is N_k, so TMA reads zeros there.
// Values are copied bit for bit; the tf32-typed tensor map rounds them on
// their way to shared memory, as it does for Q and K.
#pragma once

#include <cuda_runtime.h>

#include "fa_ptx.cuh"

#include <cstdint>

namespace fa {

struct VtParams {
  const float* V;
  long long s0, s1, s2;  // V's element strides of b, h, n (dims contiguous)
  float* Vt;
  int H_kv, N_k, dv, ldk;
  int n_kblk;            // kVtKeys-key blocks per (b, h)
};

constexpr int kVtMaxDim = 128;  // Dv of the tf32 tensor-core path
constexpr int kVtKeys = 64;     // keys per CTA

// One CTA per 64 keys of one (b, h), so that a problem of up to ~150 x 8
// blocks is read in a single wave with every load in flight at once (an
// HBM-bound pass wants bytes in flight, not threads): the 64 x Dv block goes
// through shared memory.  Loads: a warp instruction reads 4 key rows x 32
// values (four 128-byte segments), lane l taking key 4g + l / 8 and values
// c .. c + 3 with c = 32 s + 4 (l mod 8), all eight of a thread's loads
// issued before any is used (streaming loads: V is read once); the stores into the row-major tile (row stride
// kVtMaxDim + 1 = 1 mod 32 words) then fall on bank key + c + i, distinct
// over the warp.
// A 16-byte store that asks L2 to keep the line (evict-last policy).
__device__ __forceinline__ void st_evict_last(float4* dst, const float4& v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

__global__ void __launch_bounds__(256) fa_vt_kernel(const VtParams p) {
  __shared__ float tile[kVtKeys][kVtMaxDim + 1];
  // the attention kernel behind this one may start now: it waits for this
  // grid's completion before it reads V^T
  griddep_launch_dependents();
  const int bh = blockIdx.x / p.n_kblk;
  const int k0 = (blockIdx.x - bh * p.n_kblk) * kVtKeys;
  const int b = bh / p.H_kv;
  const int h = bh - b * p.H_kv;
  const float* src = p.V + b * p.s0 + h * p.s1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int segs = (p.dv + 31) >> 5;  // 32-value segments of a row
  constexpr int kGroups = kVtKeys / 4;                        // 4-key groups
  constexpr int kItems = kGroups * (kVtMaxDim / 32) / 8;      // items per warp at Dv = 128
  float4 v[kItems];
#pragma unroll
  for (int t = 0; t < kItems; ++t) {
    const int u = warp + 8 * t;  // key group + kGroups * segment
    const int key = (u % kGroups) * 4 + (lane >> 3);
    const int c = (u / kGroups) * 32 + 4 * (lane & 7);
    v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (u / kGroups < segs && k0 + key < p.N_k && c < p.dv)
      v[t] = __ldcs(reinterpret_cast<const float4*>(src + static_cast<long long>(k0 + key) * p.s2 + c));
  }
#pragma unroll
  for (int t = 0; t < kItems; ++t) {
    const int u = warp + 8 * t;
    const int key = (u % kGroups) * 4 + (lane >> 3);
    const int c = (u / kGroups) * 32 + 4 * (lane & 7);
    if (u / kGroups < segs && c < p.dv) {
      tile[key][c] = v[t].x;
      tile[key][c + 1] = v[t].y;
      tile[key][c + 2] = v[t].z;
      tile[key][c + 3] = v[t].w;
    }
  }
  __syncthreads();
  // stores: a warp instruction writes four V^T rows x 32 keys (four 128-byte
  // lines), lane l taking row c0 + l / 8 and keys 4 (l mod 8) .. + 3 of a
  // 32-key half; its four shared-memory reads tile[k + i][c] fall on bank
  // k + i + c, distinct over the warp for each i
  float* dst = p.Vt + static_cast<long long>(bh) * p.dv * p.ldk + k0;
  const int kq = 4 * (lane & 7);
  const uint64_t pol = l2_policy_evict_last();  // V^T is read again by every query tile of its head
#pragma unroll 1
  for (int c0 = 4 * warp; c0 < p.dv; c0 += 32) {
    const int c = c0 + (lane >> 3);
#pragma unroll
    for (int half = 0; half < kVtKeys / 32; ++half) {
      const int k = half * 32 + kq;
      if (c < p.dv && k0 + k < p.N_k) {
        const float4 w = make_float4(tile[k][c], tile[k + 1][c], tile[k + 2][c], tile[k + 3][c]);
        // keys past N_k (at most 3, inside the 32-key padding of ldk) are written too
        st_evict_last(reinterpret_cast<float4*>(dst + static_cast<long long>(c) * p.ldk + k), w, pol);
      }
    }
  }
}

}  // namespace fa
