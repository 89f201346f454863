// Log-sum-exp merge of n partial softmax states of one output row, spread over a CTA.
//
// Partial i covers a disjoint set of keys and holds (O_i, lse_i), where O_i is
// normalised over its keys. With M = max_i lse_i and w_i = exp(lse_i - M):
//   out = sum_i w_i O_i / sum_i w_i,   lse = M + ln sum_i w_i.
// FlashDecoding computes the partials independently and combines them all at the
// end ("【FlashAttention-V4，非官方】FlashDecoding++", section 1). No partial
// (n = 0, or every lse = -inf) gives out = 0 and lse = -inf. A NaN partial gives NaN.
//
// Warp w takes partials w, w + NW, ..., and each lane owns D/32 columns; a warp's
// loads are independent, so they are all in flight at once. The warps then
// combine through shared memory.
#pragma once

#include <cuda_bf16.h>

#include <cmath>

#include "ptx.cuh"

namespace pkv {

template <typename T>
__device__ __forceinline__ T merge_cast(float x);
template <>
__device__ __forceinline__ float merge_cast<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 merge_cast<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// `lse_of(i)` and `o_of(i)` give partial i's lse and a pointer to its D floats
// (16-byte aligned). Called by all NW*32 threads of the CTA with the same arguments.
template <typename T, int D, int NW, typename LseF, typename OF>
__device__ __forceinline__ void merge_row_cta(int n, LseF lse_of, OF o_of, T* out, float* lse_out) {
  constexpr int DL = D / 32;
  constexpr float kL2e = 1.4426950408889634f;
  __shared__ float s_acc[NW][D];
  __shared__ float s_l[NW];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  float M = -INFINITY;
  for (int i = lane; i < n; i += 32) M = fmaxf(M, lse_of(i));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (n == 0 || M == -INFINITY) {  // same on every warp
    for (int d = threadIdx.x; d < D; d += NW * 32) out[d] = merge_cast<T>(0.0f);
    if (lse_out && threadIdx.x == 0) *lse_out = -INFINITY;
    return;
  }
  float acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.0f;
  float l = 0.0f;
  int i = w;
  // up to four partials per round, loads issued before any is used
  for (; i + 3 * NW < n; i += 4 * NW) {
    float x[4][DL], wt[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      wt[k] = lse_of(i + k * NW);
      const float* o = o_of(i + k * NW) + lane * DL;
#pragma unroll
      for (int e = 0; e < DL; ++e) x[k][e] = o[e];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float wk = ex2((wt[k] - M) * kL2e);
      l += wk;
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[e] = fmaf(wk, x[k][e], acc[e]);
    }
  }
  for (; i < n; i += NW) {
    const float wk = ex2((lse_of(i) - M) * kL2e);
    const float* o = o_of(i) + lane * DL;
    l += wk;
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = fmaf(wk, o[e], acc[e]);
  }
#pragma unroll
  for (int e = 0; e < DL; ++e) s_acc[w][lane * DL + e] = acc[e];
  if (lane == 0) s_l[w] = l;
  __syncthreads();
  float L = 0.0f;
#pragma unroll
  for (int k = 0; k < NW; ++k) L += s_l[k];
  const float inv = 1.0f / L;
  for (int d = threadIdx.x; d < D; d += NW * 32) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < NW; ++k) s += s_acc[k][d];
    out[d] = merge_cast<T>(s * inv);
  }
  if (lse_out && threadIdx.x == 0) *lse_out = M + logf(L);
}

}  // namespace pkv
