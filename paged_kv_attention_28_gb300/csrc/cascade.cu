// Cascade (shared-prefix) decode: the prefix is attended once per KV head for every
// request (tensor-core kernel in prefill.cu), each request's own suffix is attended
// by the paged decode kernel, and one merge combines the partial softmax states.
//
// Two readings meet here: "级联推理" splits attention into stages that each
// handle part of the data (FlashInfer page, sections 2 and 4), and prefix
// sharing in the paged cache ("快速注意力内核与算子融合", Q&A on paged attention).
// The combination is the log-sum-exp merge of partial states that FlashDecoding
// performs at the end ("【FlashAttention-V4，非官方】FlashDecoding++", section 1).
#include <mutex>
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace pkv {
namespace {


// One warp per (request, query head) row, eight rows per CTA: combines the prefix
// chunks' and the suffix splits' partial states by log-sum-exp (merge_row_warp).
constexpr int kCascadeMergeWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kCascadeMergeWarps * 32) cascade_merge_kernel(const CascadeArgs a) {
  const int row = blockIdx.x * kCascadeMergeWarps + (threadIdx.x >> 5);
  const int rows = a.n_requests * a.n_qo_heads;
  if (row >= rows) return;
  const int r = row / a.n_qo_heads;
  const int P = a.page_size;
  const int n_pre = a.prefix_len > 0 ? a.prefix_chunks : 0;
  const int L = __ldg(a.suffix_lens + r);
  T* out = static_cast<T*>(a.out) + (size_t)row * D;
  if (L < 0 || L > a.max_suffix_blocks * P) {  // the decode kernel flagged it
    for (int d = threadIdx.x & 31; d < D; d += 32) out[d] = merge_cast<T>(NAN);
    if (a.lse && (threadIdx.x & 31) == 0) a.lse[row] = NAN;
    return;
  }
  const int nblk = (L + P - 1) / P;
  const int n_suf = (nblk + a.suffix_pages_per_split - 1) / a.suffix_pages_per_split;
  // partial i < n_pre: prefix chunk i; otherwise suffix split i - n_pre
  merge_row_warp<T, D>(
      n_pre + n_suf,
      [&](int i) {
        return i < n_pre ? a.pre_lse[(size_t)i * rows + row]
                         : a.suf_lse[(size_t)row * a.suffix_splits + (i - n_pre)];
      },
      [&](int i) {
        return i < n_pre ? a.pre_o + ((size_t)i * rows + row) * D
                         : a.suf_o + ((size_t)row * a.suffix_splits + (i - n_pre)) * D;
      },
      out, a.lse ? a.lse + row : nullptr);
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
  // The CUDA-core suffix path runs the prefix beside the suffix decode with one item per SM
  // at most. The tensor-core path starts the suffix while the prefix runs, and each suffix
  // unit merges every prefix chunk itself: about 30 % of the SMs for the prefix there, and
  // at most 8 chunks (measured on 64 requests over a 4096-token prefix, 8 KV heads: 4 to 6
  // chunks 48.5 us, 7 chunks 49.7, 8 50.0, 11 54.2). At least two key tiles per chunk
  // either way.
  const bool tc = cascade_uses_tc(n_qo_heads, n_kv_heads, 128, page_size, PKV_BF16);
  long want = (tc ? (3 * sms) / 10 : sms) / ((long)n_kv_heads * row_pairs);
  if (tc && want > 8) want = 8;
  const long max_chunks = (n_tiles + 1) / 2;
  if (want > max_chunks) want = max_chunks;
  if (want < 1) want = 1;
  const int tpc = (int)((n_tiles + want - 1) / want);
  return (n_tiles + tpc - 1) / tpc;
}

bool cascade_uses_tc(int n_qo_heads, int n_kv_heads, int head_dim, int page_size, int dtype) {
  DecodeArgs d{};
  d.n_qo_heads = n_qo_heads;
  d.n_kv_heads = n_kv_heads;
  d.head_dim = head_dim;
  d.page_size = page_size;
  d.dtype = dtype;
  return n_kv_heads > 0 && n_qo_heads % n_kv_heads == 0 && decode_tc_supported(d);
}

SplitPlan cascade_suffix_plan(int n_requests, int max_suffix_blocks, int n_qo_heads,
                              int n_kv_heads, int head_dim, int dtype) {
  // Tensor-core suffix: one unit per (request, KV head) over all its pages, which merges
  // the prefix chunks itself.
  if (cascade_uses_tc(n_qo_heads, n_kv_heads, head_dim, 16, dtype)) return SplitPlan{1, max_suffix_blocks};
  SplitPlan p = plan_decode_splits(n_requests, max_suffix_blocks, n_kv_heads, 0,
                                   decode_ctas_per_sm(dtype, head_dim, n_qo_heads / n_kv_heads));
  // Suffix lengths vary widely from request to request, and the merge that follows
  // takes the partial states anyway: cap a split at 16 pages so the CTAs stay short
  // and the last wave stays full.
  if (p.pages_per_split > 16) {
    const int S = (max_suffix_blocks + 15) / 16;
    p = plan_decode_splits(n_requests, max_suffix_blocks, n_kv_heads, S, 1);
  }
  return p;
}

namespace {

// A side stream and two events per device, created once and kept for the life of the
// process: the prefix kernel runs on the side stream beside the suffix decode, joined
// back into the caller's stream by events (which also works inside a stream capture).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

int side_stream_for_current_device(SideStream** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream& ss = g_side[dev];
  if (!ss.s) {
    if (check_launch(cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != PKV_OK ||
        check_launch(cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != PKV_OK ||
        check_launch(cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != PKV_OK)
      return PKV_ERR_LAUNCH;
  }
  *out = &ss;
  return PKV_OK;
}

}  // namespace

int launch_cascade(const CascadeArgs& a, cudaStream_t stream) {
  if (cascade_uses_tc(a.n_qo_heads, a.n_kv_heads, a.head_dim, a.page_size, a.dtype) && a.suffix_splits == 1) {
    // 1) the shared prefix, once per KV head for all requests (tensor cores), on the stream;
    // 2) each request's suffix on the tensor-core decode, launched to overlap the prefix
    //    kernel's end; each unit merges the prefix chunks with its own state and writes the
    //    final rows (no side stream, no merge launch).
    if (a.prefix_len > 0) {
      const int rc = launch_cascade_prefix(a, stream);
      if (rc != PKV_OK) return rc;
    }
    DecodeArgs d{};
    d.q = a.q;
    d.k_pages = a.k_pages;
    d.v_pages = a.v_pages;
    d.block_table = a.suffix_table;
    d.kv_lens = a.suffix_lens;
    d.out = a.out;
    d.lse = a.lse;
    d.err_flag = a.err_flag;
    d.batch = a.n_requests;
    d.max_blocks = a.max_suffix_blocks;
    d.num_pages = a.num_pages;
    d.n_qo_heads = a.n_qo_heads;
    d.n_kv_heads = a.n_kv_heads;
    d.head_dim = a.head_dim;
    d.page_size = a.page_size;
    d.num_splits = 1;
    d.pages_per_split = a.max_suffix_blocks;
    d.scale = a.scale;
    d.dtype = a.dtype;
    if (a.prefix_len > 0) {
      d.pre_o = a.pre_o;
      d.pre_lse = a.pre_lse;
      d.pre_n = a.prefix_chunks;
    }
    return launch_decode_tc(d, stream);
  }
  // 1) the shared prefix, once per KV head for all requests (tensor cores), on the side
  //    stream: it uses few CTAs, and the suffix decode below fills the other SMs.
  SideStream* side = nullptr;
  if (a.prefix_len > 0) {
    int rc = side_stream_for_current_device(&side);
    if (rc != PKV_OK) return rc;
    // One cascade at a time may use the side stream's events.
    std::lock_guard<std::mutex> lock(g_side_mu);
    if (check_launch(cudaEventRecord(side->fork, stream)) != PKV_OK ||
        check_launch(cudaStreamWaitEvent(side->s, side->fork, 0)) != PKV_OK)
      return PKV_ERR_LAUNCH;
    rc = launch_cascade_prefix(a, side->s);
    if (rc != PKV_OK) return rc;
    if (check_launch(cudaEventRecord(side->join, side->s)) != PKV_OK) return PKV_ERR_LAUNCH;
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
  if (side && check_launch(cudaStreamWaitEvent(stream, side->join, 0)) != PKV_OK) return PKV_ERR_LAUNCH;
  // 3) merge
  const int rows = a.n_requests * a.n_qo_heads;
  if (a.head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const int blocks = (rows + kCascadeMergeWarps - 1) / kCascadeMergeWarps;
  if (a.dtype == PKV_BF16)
    cascade_merge_kernel<__nv_bfloat16, 128><<<blocks, kCascadeMergeWarps * 32, 0, stream>>>(a);
  else
    cascade_merge_kernel<float, 128><<<blocks, kCascadeMergeWarps * 32, 0, stream>>>(a);
  return check_launch(cudaGetLastError());
}

}  // namespace pkv
