// Cascade (shared-prefix) decode: the prefix is attended once per KV head for every
// request (tensor-core kernel in prefill.cu), each request's own suffix is attended
// by the paged decode kernel, and one merge combines the partial softmax states.
//
// Two readings meet here: "级联推理" splits attention into stages that each
// handle part of the data (FlashInfer page, sections 2 and 4), and prefix
// sharing in the paged cache ("快速注意力内核与算子融合", Q&A on paged attention).
// The combination is the log-sum-exp merge of partial states that FlashDecoding
// performs at the end ("【FlashAttention-V4，非官方】FlashDecoding++", section 1).
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr float kLog2eC = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ T from_f32c(float x);
template <>
__device__ __forceinline__ float from_f32c<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32c<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// One warp per (request, query head) row: combines the prefix chunks' and the
// suffix splits' partial states, M = max lse, w = exp(lse - M),
// out = sum w O / sum w, lse = M + ln sum w.
template <typename T, int D>
__global__ void __launch_bounds__(128) cascade_merge_kernel(const CascadeArgs a) {
  constexpr int DL = D / 32;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int rows = a.n_requests * a.n_qo_heads;
  if (row >= rows) return;
  const int r = row / a.n_qo_heads;
  const int P = a.page_size;
  const int n_pre = a.prefix_len > 0 ? a.prefix_chunks : 0;
  const int L = __ldg(a.suffix_lens + r);
  T* out = static_cast<T*>(a.out) + (size_t)row * D + lane * DL;
  if (L < 0 || L > a.max_suffix_blocks * P) {  // the decode kernel flagged it
#pragma unroll
    for (int e = 0; e < DL; ++e) out[e] = from_f32c<T>(NAN);
    if (a.lse && lane == 0) a.lse[row] = NAN;
    return;
  }
  const int nblk = (L + P - 1) / P;
  const int n_suf = (nblk + a.suffix_pages_per_split - 1) / a.suffix_pages_per_split;
  // part i < n_pre: prefix chunk i; otherwise suffix split i - n_pre
  auto part_lse = [&](int i) -> float {
    return i < n_pre ? a.pre_lse[(size_t)i * rows + row]
                     : a.suf_lse[(size_t)row * a.suffix_splits + (i - n_pre)];
  };
  auto part_o = [&](int i) -> const float* {
    return i < n_pre ? a.pre_o + ((size_t)i * rows + row) * D
                     : a.suf_o + ((size_t)row * a.suffix_splits + (i - n_pre)) * D;
  };
  const int n = n_pre + n_suf;
  float M = -INFINITY;
  for (int i = lane; i < n; i += 32) M = fmaxf(M, part_lse(i));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (n == 0 || M == -INFINITY) {
#pragma unroll
    for (int e = 0; e < DL; ++e) out[e] = from_f32c<T>(0.0f);
    if (a.lse && lane == 0) a.lse[row] = -INFINITY;
    return;
  }
  float acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.0f;
  float Ls = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float w = ex2((part_lse(i) - M) * kLog2eC);
    Ls += w;
    const float* o = part_o(i) + lane * DL;
    if constexpr (DL == 4) {
      const float4 x = *reinterpret_cast<const float4*>(o);
      acc[0] = fmaf(w, x.x, acc[0]);
      acc[1] = fmaf(w, x.y, acc[1]);
      acc[2] = fmaf(w, x.z, acc[2]);
      acc[3] = fmaf(w, x.w, acc[3]);
    } else {
#pragma unroll
      for (int e = 0; e < DL; ++e) acc[e] = fmaf(w, o[e], acc[e]);
    }
  }
  const float inv = 1.0f / Ls;
#pragma unroll
  for (int e = 0; e < DL; ++e) out[e] = from_f32c<T>(acc[e] * inv);
  if (a.lse && lane == 0) a.lse[row] = M + logf(Ls);
}

}  // namespace

int cascade_prefix_chunks(int prefix_len, int page_size, int n_requests, int n_qo_heads,
                          int n_kv_heads) {
  if (prefix_len <= 0 || page_size <= 0) return 0;
  const int n_pages = (prefix_len + page_size - 1) / page_size;
  const int n_tiles = (n_pages + 7) / 8;  // 128-key tiles of 8 pages of 16
  const int G = n_qo_heads / n_kv_heads;
  const long row_pairs = ((long)n_requests * G + 255) / 256;
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  // About half the SMs for the prefix, and at least four key tiles per chunk so that
  // each CTA's query load and partial-state write are amortised.
  long want = (sms / 2) / ((long)n_kv_heads * row_pairs);
  const long max_chunks = (n_tiles + 3) / 4;
  if (want > max_chunks) want = max_chunks;
  if (want < 1) want = 1;
  const int tpc = (int)((n_tiles + want - 1) / want);
  return (n_tiles + tpc - 1) / tpc;
}

SplitPlan cascade_suffix_plan(int n_requests, int max_suffix_blocks, int n_qo_heads,
                              int n_kv_heads, int head_dim, int dtype) {
  return plan_decode_splits(n_requests, max_suffix_blocks, n_kv_heads, 0,
                            decode_ctas_per_sm(dtype, head_dim, n_qo_heads / n_kv_heads));
}

int launch_cascade(const CascadeArgs& a, cudaStream_t stream) {
  // 1) the shared prefix, once per KV head for all requests (tensor cores)
  if (a.prefix_len > 0) {
    const int rc = launch_cascade_prefix(a, stream);
    if (rc != PKV_OK) return rc;
  }
  // 2) every request's own suffix pages: fp32 partial states, one per live split
  DecodeArgs d{};
  d.q = a.q;
  d.k_pages = a.k_pages;
  d.v_pages = a.v_pages;
  d.block_table = a.suffix_table;
  d.kv_lens = a.suffix_lens;
  d.part_o = a.suf_o;
  d.part_lse = a.suf_lse;
  d.err_flag = a.err_flag;
  d.batch = a.n_requests;
  d.max_blocks = a.max_suffix_blocks;
  d.num_pages = a.num_pages;
  d.n_qo_heads = a.n_qo_heads;
  d.n_kv_heads = a.n_kv_heads;
  d.head_dim = a.head_dim;
  d.page_size = a.page_size;
  d.num_splits = a.suffix_splits;
  d.pages_per_split = a.suffix_pages_per_split;
  d.scale = a.scale;
  d.dtype = a.dtype;
  d.partial_only = true;
  int rc = launch_decode_partials(d, stream);
  if (rc != PKV_OK) return rc;
  // 3) merge
  const int rows = a.n_requests * a.n_qo_heads;
  if (a.head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (a.dtype == PKV_BF16)
    cascade_merge_kernel<__nv_bfloat16, 128><<<(rows + 3) / 4, 128, 0, stream>>>(a);
  else
    cascade_merge_kernel<float, 128><<<(rows + 3) / 4, 128, 0, stream>>>(a);
  return check_launch(cudaGetLastError());
}

}  // namespace pkv
