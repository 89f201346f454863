// Host-side declarations shared by the launch layer and the kernel files.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "pkv_attn.h"

namespace pkv {

// Everything a decode launch needs (device pointers and resolved sizes).
struct DecodeArgs {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* block_table;
  const int32_t* kv_lens;
  void* out;
  float* lse;
  float* part_o;    // [batch][n_qo_heads][num_splits][head_dim], used when num_splits > 1
  float* part_lse;  // [batch][n_qo_heads][num_splits]
  int32_t* err_flag;
  int batch, max_blocks, num_pages, n_qo_heads, n_kv_heads, head_dim, page_size;
  int num_splits, pages_per_split;
  float scale;
  int dtype;
  // every live split writes an fp32 partial state, even a sequence's only split
  // (used by the cascade path, whose own merge combines them with the prefix)
  bool partial_only;
  // unified-max variant
  bool unified;
  float phi;
  int32_t* fallback_count;
  // FP8 E4M3 page pools (q and out are bf16): one scale per (page, KV head) of K and V
  bool fp8;
  const float* k_scale;  // [num_pages][n_kv_heads]
  const float* v_scale;
  // Stall injection for the failure-handling test (attn_debug_decode_stall): the producer
  // of every CTA withholds the copies of page `stall_page` of its split (-1: none), and
  // every bounded wait gives up after wait_limit_ns.
  int stall_page = -1;
  uint64_t wait_limit_ns = 2000000000ull;  // the default limit of every bounded wait
  // Cascade (tensor-core decode only): the shared prefix's fp32 partial states, pre_n chunks
  // of O [pre_n][batch][n_qo_heads][head_dim] and LSE [pre_n][batch][n_qo_heads], written by
  // the kernel launched just before on the same stream. Each sequence (one split) merges them
  // with its own state and writes the final rows; the launch overlaps the prefix kernel's end
  // (programmatic dependent launch) and waits for it before reading these.
  const float* pre_o = nullptr;
  const float* pre_lse = nullptr;
  int pre_n = 0;
};


// The stall injection that decode launches pick up (process-wide; off by default).
void decode_stall_settings(int* page, uint64_t* wait_limit_ns);

struct SplitPlan {
  int num_splits;
  int pages_per_split;
};

int device_sm_count();

// The dynamic shared-memory limit of one kernel, raised once per device before its first
// launch there. A device's bit is set only after the attribute call has succeeded, so a
// thread that sees it set launches on a configured kernel; two threads making a first call
// at the same time may both set the attribute, which is harmless.
struct FuncConfigured {
  std::atomic<uint64_t> mask{0};  // one bit per device ordinal < 64
  bool ensure(const void* func, int smem_bytes);
};

// Remembers the most recent failing CUDA call of this host thread (see
// attn_last_cuda_error_string) and returns PKV_ERR_LAUNCH, or PKV_OK on success.
int check_launch(cudaError_t e);
// Split count and pages per split. `ctas_per_sm` is how many decode CTAs of the
// dispatched instantiation fit on one SM (decode_ctas_per_sm).
SplitPlan plan_decode_splits(int batch, int max_blocks, int n_kv_heads, int requested,
                             int ctas_per_sm);
int decode_ctas_per_sm(int dtype, int head_dim, int group);

// Enqueues the decode kernel (and the merge kernel when num_splits > 1).
int launch_decode(const DecodeArgs& a, cudaStream_t stream);
// Enqueues only the decode kernel (the caller merges the partial states).
int launch_decode_partials(const DecodeArgs& a, cudaStream_t stream);
bool decode_supported(int dtype, int head_dim, int page_size, int group);
// The tensor-core decode (decode_tc.cu): bf16, head_dim 128, page 16, groups of 4 or 8.
bool decode_tc_supported(const DecodeArgs& a);
int launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);

int launch_merge_pair(const float* out_a, const float* lse_a, const float* out_b,
                      const float* lse_b, void* out, float* lse, int n_rows, int head_dim,
                      int out_dtype, cudaStream_t stream);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int32_t* err_flag;
  int batch, seq_len, n_qo_heads, n_kv_heads, head_dim;
  float scale;
};
int launch_prefill(const PrefillArgs& a, cudaStream_t stream);

struct CascadeArgs {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* prefix_table;
  int prefix_len;
  const int32_t* suffix_table;
  const int32_t* suffix_lens;
  void* out;
  float* lse;
  int n_requests, max_suffix_blocks, num_pages, n_qo_heads, n_kv_heads, head_dim, page_size;
  float scale;
  int dtype;
  int32_t* err_flag;
  // workspace carve-up
  float* pre_o;     // [prefix_chunks][n_requests][n_qo_heads][head_dim]
  float* pre_lse;   // [prefix_chunks][n_requests][n_qo_heads]
  float* suf_o;     // [n_requests][n_qo_heads][suffix_splits][head_dim]
  float* suf_lse;   // [n_requests][n_qo_heads][suffix_splits]
  int prefix_chunks;
  int suffix_splits, suffix_pages_per_split;
};
// Chunks the shared prefix is cut into (0 when there is no prefix), from the shape
// and the SM count of the current device.
int cascade_prefix_chunks(int prefix_len, int page_size, int n_requests, int n_qo_heads,
                          int n_kv_heads);
SplitPlan cascade_suffix_plan(int n_requests, int max_suffix_blocks, int n_qo_heads,
                              int n_kv_heads, int head_dim, int dtype);
// True when the cascade's suffix runs on the tensor-core decode and merges the prefix there.
bool cascade_uses_tc(int n_qo_heads, int n_kv_heads, int head_dim, int page_size, int dtype);
int launch_cascade_prefix(const CascadeArgs& a, cudaStream_t stream);

struct ChunkArgs {
  const void* q;        // bf16 [batch][chunk_len][n_qo_heads][head_dim]
  const void* k_pages;  // bf16 [num_pages][n_kv_heads][page_size][head_dim]
  const void* v_pages;
  const int32_t* block_table;  // [batch][max_blocks]
  const int32_t* prefix_lens;  // [batch]
  void* out;                   // bf16 [batch][chunk_len][n_qo_heads][head_dim]
  float* lse;                  // fp32 [batch][n_qo_heads][chunk_len] (nullable)
  int32_t* err_flag;
  int batch, chunk_len, max_blocks, num_pages, n_qo_heads, n_kv_heads, head_dim, page_size;
  float scale;
};
int launch_prefill_chunk(const ChunkArgs& a, cudaStream_t stream);

// Flat GEMM of the decode phase: y[m][n] = sum_k x[m][k] * w[n][k], bf16 in and out.
struct FlatGemmArgs {
  const void* x;  // bf16 [m][k]
  const void* w;  // bf16 [n][k]
  void* y;        // bf16 [m][n]
  int32_t* err_flag;
  int m, n, k;
};
struct FlatGemmPlan {
  int tiles;       // 128-row tiles of w
  int splits;      // CTAs per tile (a cluster) that share K
  int kc_per_cta;  // 64-column slices of K per CTA
  int n_kc;        // 64-column slices of K in all
};
constexpr int kFlatGemmMaxM = 64;
int flat_gemm_padded_m(int m);
FlatGemmPlan plan_flat_gemm(int m, int n, int k);
int launch_flat_gemm(const FlatGemmArgs& a, cudaStream_t stream);
int launch_cascade(const CascadeArgs& a, cudaStream_t stream);

}  // namespace pkv
