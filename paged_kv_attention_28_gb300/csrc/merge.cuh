// Log-sum-exp merge of n partial softmax states of one output row, by one warp.
//
// Partial i covers a disjoint set of keys and holds (O_i, lse_i), where O_i is
// normalised over its keys. With M = max_i lse_i and w_i = exp(lse_i - M):
//   out = sum_i w_i O_i / sum_i w_i,   lse = M + ln sum_i w_i.
// FlashDecoding computes the partials independently and combines them all at the
// end ("【FlashAttention-V4，非官方】FlashDecoding++", section 1). No partial
// (n = 0, or every lse = -inf) gives out = 0 and lse = -inf. A NaN partial gives NaN.
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

// DL consecutive floats from a 4*DL-byte aligned address, in one load where DL is 2 or 4.
template <int DL>
__device__ __forceinline__ void load_cols(const float* p, float (&x)[DL]) {
  if constexpr (DL == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
  } else if constexpr (DL == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x, x[1] = v.y;
  } else {
#pragma unroll
    for (int e = 0; e < DL; ++e) x[e] = p[e];
  }
}

// `lse_of(i)` and `o_of(i)` give partial i's lse and a pointer to its D floats
// (16-byte aligned); every lane of the warp calls this with the same arguments. Lane l
// owns columns [l*D/32, (l+1)*D/32). Every lane computes the weights itself (the lse
// loads are broadcasts), and the partials' loads are issued eight (then four) at a time
// before any is used. No shared memory and no CTA barrier, so a CTA can hold one row per warp.
template <typename T, int D, typename LseF, typename OF>
__device__ __forceinline__ void merge_row_warp(int n, LseF lse_of, OF o_of, T* out, float* lse_out) {
  constexpr int DL = D / 32;
  constexpr float kL2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  float M = -INFINITY;
  bool bad = false;  // a NaN partial (a failed split); fmaxf alone would skip it
  for (int i = lane; i < n; i += 32) {
    const float x = lse_of(i);
    bad |= x != x;
    M = fmaxf(M, x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  T* o_row = out + lane * DL;
  if (__any_sync(0xffffffffu, bad)) {
#pragma unroll
    for (int e = 0; e < DL; ++e) o_row[e] = merge_cast<T>(NAN);
    if (lse_out && lane == 0) *lse_out = NAN;
    return;
  }
  if (n == 0 || M == -INFINITY) {
#pragma unroll
    for (int e = 0; e < DL; ++e) o_row[e] = merge_cast<T>(0.0f);
    if (lse_out && lane == 0) *lse_out = -INFINITY;
    return;
  }
  float acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.0f;
  float l = 0.0f;
  int i = 0;
  for (; i + 7 < n; i += 8) {
    float x[8][DL], wt[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      wt[k] = lse_of(i + k);
      load_cols<DL>(o_of(i + k) + lane * DL, x[k]);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float wk = ex2((wt[k] - M) * kL2e);
      l += wk;
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[e] = fmaf(wk, x[k][e], acc[e]);
    }
  }
  for (; i + 3 < n; i += 4) {
    float x[4][DL], wt[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      wt[k] = lse_of(i + k);
      load_cols<DL>(o_of(i + k) + lane * DL, x[k]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float wk = ex2((wt[k] - M) * kL2e);
      l += wk;
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[e] = fmaf(wk, x[k][e], acc[e]);
    }
  }
  for (; i < n; ++i) {
    const float wk = ex2((lse_of(i) - M) * kL2e);
    float x[DL];
    load_cols<DL>(o_of(i) + lane * DL, x);
    l += wk;
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = fmaf(wk, x[e], acc[e]);
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int e = 0; e < DL; ++e) o_row[e] = merge_cast<T>(acc[e] * inv);
  if (lse_out && lane == 0) *lse_out = M + logf(l);
}

// The same merge by the MW warps of a CTA, for rows with many partials: warp w takes
// partials w, w + MW, ... eight at a time, all eight loads in flight before any is used,
// keeps its own running (max, sum, weighted O), and the warps' states are combined through
// shared memory. For n <= 8 MW every load of the row is issued in one round. Every thread
// of the CTA calls this with the same arguments; `sm` holds MW * (D + 3) floats.
template <typename T, int D, int MW, typename LseF, typename OF>
__device__ __forceinline__ void merge_row_cta(int n, LseF lse_of, OF o_of, T* out, float* lse_out, float* sm) {
  constexpr int DL = D / 32, PER = 8;
  constexpr float kL2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = -INFINITY, l = 0.0f, acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.0f;
  bool bad = false;
  for (int base = warp; base < n; base += MW * PER) {
    float w[PER], x[PER][DL];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = base + k * MW;
      if (i < n) {
        w[k] = lse_of(i);
        load_cols<DL>(o_of(i) + lane * DL, x[k]);
      } else {
        w[k] = -INFINITY;
#pragma unroll
        for (int e = 0; e < DL; ++e) x[k][e] = 0.0f;
      }
    }
    float mn = m;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      bad |= w[k] != w[k];
      mn = fmaxf(mn, w[k]);
    }
    if (mn == -INFINITY) continue;
    const float sc = ex2((m - mn) * kL2e);  // 0 while m = -inf
    l *= sc;
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] *= sc;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const float wk = ex2((w[k] - mn) * kL2e);  // 0 for the slots past n
      l += wk;
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[e] = fmaf(wk, x[k][e], acc[e]);
    }
    m = mn;
  }
  float* s_acc = sm;               // [MW][D]
  float* s_m = sm + MW * D;        // [MW]
  float* s_l = s_m + MW;           // [MW]
  float* s_bad = s_l + MW;         // [MW]
#pragma unroll
  for (int e = 0; e < DL; ++e) s_acc[warp * D + lane * DL + e] = acc[e];
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
    s_bad[warp] = bad ? 1.0f : 0.0f;
  }
  __syncthreads();
  float M = -INFINITY, nan_seen = 0.0f;
#pragma unroll
  for (int v = 0; v < MW; ++v) {
    M = fmaxf(M, s_m[v]);
    nan_seen += s_bad[v];
  }
  float sc[MW], L = 0.0f;
#pragma unroll
  for (int v = 0; v < MW; ++v) {
    sc[v] = M == -INFINITY ? 0.0f : ex2((s_m[v] - M) * kL2e);
    L = fmaf(sc[v], s_l[v], L);
  }
  for (int c = threadIdx.x; c < D; c += MW * 32) {
    float o = 0.0f;
#pragma unroll
    for (int v = 0; v < MW; ++v) o = fmaf(sc[v], s_acc[v * D + c], o);
    out[c] = merge_cast<T>(nan_seen > 0.0f ? NAN : M == -INFINITY ? 0.0f : o / L);
  }
  if (lse_out && threadIdx.x == 0) *lse_out = nan_seen > 0.0f ? NAN : M == -INFINITY ? -INFINITY : M + logf(L);
}

}  // namespace pkv
