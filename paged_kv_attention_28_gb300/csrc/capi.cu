// C ABI: argument checks, split planning, workspace sizing and dispatch.
// No call allocates, frees, copies to the host or synchronises.
#include <cmath>
#include <cstdint>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace pkv {

// An NVTX range around each compute call, named after the call, so that a trace (Nsight
// Systems, or ncu with --nvtx) shows which library call launched which kernels. Without a
// tool attached an NVTX call only tests a function pointer.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

static thread_local cudaError_t g_last_error = cudaSuccess;

int check_launch(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  g_last_error = e;
  return PKV_ERR_LAUNCH;
}

int device_sm_count() {
  static std::atomic<int> cache[64];  // zero-initialised (static storage); 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_release);
  return n;
}

namespace {
std::atomic<int> g_stall_page{-1};
std::atomic<uint64_t> g_stall_limit_ns{0};
}  // namespace

void decode_stall_settings(int* page, uint64_t* wait_limit_ns) {
  *page = g_stall_page.load(std::memory_order_relaxed);
  const uint64_t lim = g_stall_limit_ns.load(std::memory_order_relaxed);
  if (lim > 0) *wait_limit_ns = lim;
}

bool FuncConfigured::ensure(const void* func, int smem_bytes) {
  int dev = 0;
  if (check_launch(cudaGetDevice(&dev)) != PKV_OK) return false;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit && (mask.load(std::memory_order_acquire) & bit)) return true;
  if (check_launch(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes)) !=
      PKV_OK)
    return false;
  if (bit) mask.fetch_or(bit, std::memory_order_release);
  return true;
}

SplitPlan plan_decode_splits(int batch, int max_blocks, int n_kv_heads, int requested,
                             int ctas_per_sm) {
  int S;
  if (requested > 0) {
    S = requested < max_blocks ? requested : max_blocks;
  } else {
    // Model the time of a split count as (waves of CTAs) x (pages per CTA + a fixed
    // per-CTA cost of about 4 pages), assuming every sequence is full length, plus the
    // split merge when there is more than one split: one more launch, whose latency is
    // worth about 24 pages of one CTA's streaming. Take the cheapest. This favours splits
    // that fill whole waves of resident CTAs, and one split for small problems.
    constexpr long kMergePages = 24;
    int sms = device_sm_count();
    if (sms <= 0) sms = 148;
    const long slots = (long)sms * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    const long units = (long)batch * n_kv_heads;
    const int s_max = max_blocks < 64 ? max_blocks : 64;
    long best_cost = -1;
    S = 1;
    for (int s = 1; s <= s_max; ++s) {
      const long pps = (max_blocks + s - 1) / s;
      const long waves = (units * s + slots - 1) / slots;
      const long cost = waves * (pps + 4) + (s > 1 ? kMergePages : 0);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        S = s;
      }
    }
  }
  const int pps = (max_blocks + S - 1) / S;
  return SplitPlan{(max_blocks + pps - 1) / pps, pps};
}

// The split plan of a decode call, the same for the call and for the size queries. E4M3
// pools at head_dim 128 (page 16, groups of 1, 2, 4 or 8) run on the tensor-core decode and
// are planned as the bf16 ones; the others on the CUDA-core kernel, whose E4M3 CTA takes two
// KV heads.
static SplitPlan plan_decode(int batch, int max_blocks, int n_qo_heads, int n_kv_heads, int head_dim, int page_size,
                      int num_splits, int dtype) {
  const int G = n_qo_heads / n_kv_heads;
  if (dtype == PKV_FP8_E4M3) {
    DecodeArgs d{};
    d.n_qo_heads = n_qo_heads;
    d.n_kv_heads = n_kv_heads;
    d.head_dim = head_dim;
    d.page_size = page_size;
    d.dtype = PKV_BF16;
    d.fp8 = true;
    if (decode_tc_supported(d))
      return plan_decode_splits(batch, max_blocks, n_kv_heads, num_splits, decode_ctas_per_sm(PKV_BF16, head_dim, G));
    return plan_decode_splits(batch, max_blocks, n_kv_heads / 2, num_splits, decode_ctas_per_sm(dtype, head_dim, G));
  }
  return plan_decode_splits(batch, max_blocks, n_kv_heads, num_splits, decode_ctas_per_sm(dtype, head_dim, G));
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split partials: O [rows][S][D], LSE [rows][S].
static size_t decode_ws_bytes(int batch, int n_qo_heads, int n_kv_heads, int head_dim, int S) {
  (void)n_kv_heads;
  if (S <= 1) return 0;
  const size_t rows = (size_t)batch * n_qo_heads;
  return align_up(rows * S * head_dim * sizeof(float), 256) + align_up(rows * S * sizeof(float), 256);
}


static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DecodeCall {
  const void *q, *k_pages, *v_pages;
  const int32_t *block_table, *kv_lens;
  void* out;
  float* lse;
  int batch, max_blocks, num_pages, n_qo_heads, n_kv_heads, head_dim, page_size;
  float scale;
  int num_splits, dtype;
  void* workspace;
  size_t workspace_bytes;
  int32_t* err_flag;
  cudaStream_t stream;
  // FP8 page pools (dtype is then PKV_BF16, the type of q and out)
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
};

static int decode_common(const DecodeCall& c, bool unified, float phi, int32_t* fallback_count,
                         bool fp8 = false) {
  if (c.batch < 0 || c.max_blocks < 1 || c.num_pages < 1 || c.n_qo_heads < 1 ||
      c.n_kv_heads < 1 || c.head_dim < 1 || c.page_size < 1 || c.num_splits < 0)
    return PKV_ERR_INVALID_ARG;
  if (c.n_qo_heads % c.n_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(c.scale) || (unified && !std::isfinite(phi))) return PKV_ERR_INVALID_ARG;
  if (c.dtype != PKV_F32 && c.dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if ((long)c.max_blocks * c.page_size > 0x7fffffffL) return PKV_ERR_INVALID_ARG;
  if (c.batch == 0) return PKV_OK;
  if (!c.q || !c.k_pages || !c.v_pages || !c.block_table || !c.kv_lens || !c.out)
    return PKV_ERR_INVALID_ARG;
  if (fp8 && (!c.k_scale || !c.v_scale)) return PKV_ERR_INVALID_ARG;
  if (!aligned16(c.k_pages) || !aligned16(c.v_pages)) return PKV_ERR_INVALID_ARG;
  const int G = c.n_qo_heads / c.n_kv_heads;
  if (!decode_supported(c.dtype, c.head_dim, c.page_size, G)) return PKV_ERR_UNSUPPORTED;
  if (c.batch > 65535 || c.n_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (fp8 && c.n_kv_heads % 2) return PKV_ERR_UNSUPPORTED;  // two KV heads per CTA
  const SplitPlan plan = plan_decode(c.batch, c.max_blocks, c.n_qo_heads, c.n_kv_heads, c.head_dim, c.page_size,
                                     c.num_splits, fp8 ? PKV_FP8_E4M3 : c.dtype);
  const size_t need = decode_ws_bytes(c.batch, c.n_qo_heads, c.n_kv_heads, c.head_dim, plan.num_splits);
  if (need > 0 && (!c.workspace || c.workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(c.workspace) & 255u) != 0))
    return PKV_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_DEVICE;

  DecodeArgs a{};
  a.q = c.q;
  a.k_pages = c.k_pages;
  a.v_pages = c.v_pages;
  a.block_table = c.block_table;
  a.kv_lens = c.kv_lens;
  a.out = c.out;
  a.lse = c.lse;
  const size_t rows = (size_t)c.batch * c.n_qo_heads;
  if (need > 0) {
    char* w = static_cast<char*>(c.workspace);
    a.part_o = reinterpret_cast<float*>(w);
    w += align_up(rows * plan.num_splits * c.head_dim * sizeof(float), 256);
    a.part_lse = reinterpret_cast<float*>(w);
  }
  a.err_flag = c.err_flag;
  a.batch = c.batch;
  a.max_blocks = c.max_blocks;
  a.num_pages = c.num_pages;
  a.n_qo_heads = c.n_qo_heads;
  a.n_kv_heads = c.n_kv_heads;
  a.head_dim = c.head_dim;
  a.page_size = c.page_size;
  a.num_splits = plan.num_splits;
  a.pages_per_split = plan.pages_per_split;
  a.scale = c.scale;
  a.dtype = c.dtype;
  a.unified = unified;
  a.phi = phi;
  a.fallback_count = fallback_count;
  decode_stall_settings(&a.stall_page, &a.wait_limit_ns);
  a.fp8 = fp8;
  a.k_scale = c.k_scale;
  a.v_scale = c.v_scale;
  return launch_decode(a, c.stream);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_LAUNCH: return "CUDA launch failed";
    case PKV_ERR_DEVICE: return "no usable CUDA device";
    default: return "unknown status";
  }
}

const char* attn_last_cuda_error_string(void) {
  return g_last_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_error);
}

int attn_decode_num_splits(int batch, int max_blocks_per_seq, int n_qo_heads, int n_kv_heads,
                           int head_dim, int page_size, int num_splits, int dtype) {
  if (batch < 0 || max_blocks_per_seq < 1 || n_qo_heads < 1 || n_kv_heads < 1 ||
      head_dim < 1 || page_size < 1 || num_splits < 0 || n_qo_heads % n_kv_heads)
    return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F32 && dtype != PKV_BF16 && dtype != PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  if (dtype == PKV_FP8_E4M3 && n_kv_heads % 2) return PKV_ERR_UNSUPPORTED;
  return plan_decode(batch, max_blocks_per_seq, n_qo_heads, n_kv_heads, head_dim, page_size, num_splits, dtype)
      .num_splits;
}

size_t attn_decode_workspace_size(int batch, int max_blocks_per_seq, int n_qo_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_splits,
                                  int dtype) {
  const int S = attn_decode_num_splits(batch, max_blocks_per_seq, n_qo_heads, n_kv_heads,
                                       head_dim, page_size, num_splits, dtype);
  if (S < 0) return (size_t)-1;
  return decode_ws_bytes(batch, n_qo_heads, n_kv_heads, head_dim, S);
}

int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* block_table, const int32_t* kv_lens, void* out, float* lse,
                      int batch, int max_blocks_per_seq, int num_pages, int n_qo_heads,
                      int n_kv_heads, int head_dim, int page_size, float scale, int num_splits,
                      int dtype, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                      void* stream) {
  const pkv::CallRange range("attn_decode_paged");
  DecodeCall c{q, k_pages, v_pages, block_table, kv_lens, out, lse, batch, max_blocks_per_seq,
               num_pages, n_qo_heads, n_kv_heads, head_dim, page_size, scale, num_splits, dtype,
               workspace, workspace_bytes, err_flag, static_cast<cudaStream_t>(stream)};
  return decode_common(c, false, 0.0f, nullptr);
}

int attn_decode_paged_unified_max(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* kv_lens, void* out,
                                  float* lse, int batch, int max_blocks_per_seq, int num_pages,
                                  int n_qo_heads, int n_kv_heads, int head_dim, int page_size,
                                  float scale, int num_splits, int dtype, float phi,
                                  int32_t* fallback_count, void* workspace,
                                  size_t workspace_bytes, int32_t* err_flag, void* stream) {
  const pkv::CallRange range("attn_decode_paged_unified_max");
  DecodeCall c{q, k_pages, v_pages, block_table, kv_lens, out, lse, batch, max_blocks_per_seq,
               num_pages, n_qo_heads, n_kv_heads, head_dim, page_size, scale, num_splits, dtype,
               workspace, workspace_bytes, err_flag, static_cast<cudaStream_t>(stream)};
  return decode_common(c, true, phi, fallback_count);
}

int attn_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages,
                          const float* k_scale, const float* v_scale, const int32_t* block_table,
                          const int32_t* kv_lens, void* out, float* lse, int batch,
                          int max_blocks_per_seq, int num_pages, int n_qo_heads, int n_kv_heads,
                          int head_dim, int page_size, float scale, int num_splits,
                          void* workspace, size_t workspace_bytes, int32_t* err_flag,
                          void* stream) {
  const pkv::CallRange range("attn_decode_paged_fp8");
  DecodeCall c{q, k_pages, v_pages, block_table, kv_lens, out, lse, batch, max_blocks_per_seq,
               num_pages, n_qo_heads, n_kv_heads, head_dim, page_size, scale, num_splits, PKV_BF16,
               workspace, workspace_bytes, err_flag, static_cast<cudaStream_t>(stream), k_scale,
               v_scale};
  return decode_common(c, false, 0.0f, nullptr, true);
}

int attn_merge_states(const float* out_a, const float* lse_a, const float* out_b,
                      const float* lse_b, void* out, float* lse, int n_rows, int head_dim,
                      int out_dtype, void* stream) {
  const pkv::CallRange range("attn_merge_states");
  if (n_rows < 0 || head_dim < 1) return PKV_ERR_INVALID_ARG;
  if (out_dtype != PKV_F32 && out_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (n_rows == 0) return PKV_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out) return PKV_ERR_INVALID_ARG;
  if (n_rows > 65535L * 4 * 1024) return PKV_ERR_UNSUPPORTED;
  return launch_merge_pair(out_a, lse_a, out_b, lse_b, out, lse, n_rows, head_dim, out_dtype,
                           static_cast<cudaStream_t>(stream));
}

int attn_prefill_causal(const void* q, const void* k, const void* v, void* out, float* lse,
                        int batch, int seq_len, int n_qo_heads, int n_kv_heads, int head_dim,
                        float scale, int dtype, int32_t* err_flag, void* stream) {
  const pkv::CallRange range("attn_prefill_causal");
  if (batch < 0 || seq_len < 0 || n_qo_heads < 1 || n_kv_heads < 1 || head_dim < 1)
    return PKV_ERR_INVALID_ARG;
  if (n_qo_heads % n_kv_heads || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (batch == 0 || seq_len == 0) return PKV_OK;
  if (!q || !k || !v || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_BF16 || head_dim != 128) return PKV_ERR_UNSUPPORTED;
  PrefillArgs a{q, k, v, out, lse, err_flag, batch, seq_len, n_qo_heads, n_kv_heads, head_dim, scale};
  return launch_prefill(a, static_cast<cudaStream_t>(stream));
}

int attn_prefill_paged_chunk(const void* q, const void* k_pages, const void* v_pages,
                             const int32_t* block_table, const int32_t* prefix_lens, void* out,
                             float* lse, int batch, int chunk_len, int max_blocks_per_seq,
                             int num_pages, int n_qo_heads, int n_kv_heads, int head_dim,
                             int page_size, float scale, int dtype, int32_t* err_flag,
                             void* stream) {
  const pkv::CallRange range("attn_prefill_paged_chunk");
  if (batch < 0 || chunk_len < 0 || max_blocks_per_seq < 1 || num_pages < 1 || n_qo_heads < 1 ||
      n_kv_heads < 1 || head_dim < 1 || page_size < 1)
    return PKV_ERR_INVALID_ARG;
  if (n_qo_heads % n_kv_heads || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if ((long)max_blocks_per_seq * page_size > 0x7fffffffL) return PKV_ERR_INVALID_ARG;
  if (chunk_len > max_blocks_per_seq * page_size) return PKV_ERR_INVALID_ARG;
  if (batch == 0 || chunk_len == 0) return PKV_OK;
  if (!q || !k_pages || !v_pages || !block_table || !prefix_lens || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return PKV_ERR_INVALID_ARG;
  const int G = n_qo_heads / n_kv_heads;
  if (dtype != PKV_BF16 || head_dim != 128 || page_size != 16 || 128 % G) return PKV_ERR_UNSUPPORTED;
  if (batch > 65535) return PKV_ERR_UNSUPPORTED;
  ChunkArgs a{q, k_pages, v_pages, block_table, prefix_lens, out, lse, err_flag, batch, chunk_len,
              max_blocks_per_seq, num_pages, n_qo_heads, n_kv_heads, head_dim, page_size, scale};
  return launch_prefill_chunk(a, static_cast<cudaStream_t>(stream));
}

size_t attn_cascade_workspace_size(int n_requests, int prefix_len, int max_suffix_blocks,
                                   int n_qo_heads, int n_kv_heads, int head_dim, int page_size) {
  if (n_requests < 0 || prefix_len < 0 || max_suffix_blocks < 1 || n_qo_heads < 1 ||
      n_kv_heads < 1 || head_dim < 1 || page_size < 1 || n_qo_heads % n_kv_heads)
    return (size_t)-1;
  const size_t rows = (size_t)n_requests * n_qo_heads;
  const int chunks = cascade_prefix_chunks(prefix_len, page_size, n_requests, n_qo_heads, n_kv_heads);
  const SplitPlan suf = cascade_suffix_plan(n_requests, max_suffix_blocks, n_qo_heads, n_kv_heads,
                                            head_dim, PKV_BF16);
  return align_up((size_t)chunks * rows * head_dim * 4, 256) + align_up((size_t)chunks * rows * 4, 256) +
         align_up(rows * suf.num_splits * head_dim * 4, 256) + align_up(rows * suf.num_splits * 4, 256);
}

int attn_decode_cascade(const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* prefix_block_table, int prefix_len,
                        const int32_t* suffix_block_table, const int32_t* suffix_lens, void* out,
                        float* lse, int n_requests, int max_suffix_blocks, int num_pages,
                        int n_qo_heads, int n_kv_heads, int head_dim, int page_size, float scale,
                        int dtype, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                        void* stream) {
  const pkv::CallRange range("attn_decode_cascade");
  if (n_requests < 0 || prefix_len < 0 || max_suffix_blocks < 1 || num_pages < 1 ||
      n_qo_heads < 1 || n_kv_heads < 1 || head_dim < 1 || page_size < 1)
    return PKV_ERR_INVALID_ARG;
  if (n_qo_heads % n_kv_heads || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (n_requests == 0) return PKV_OK;
  if (!q || !k_pages || !v_pages || !suffix_block_table || !suffix_lens || !out)
    return PKV_ERR_INVALID_ARG;
  if (prefix_len > 0 && !prefix_block_table) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages)) return PKV_ERR_INVALID_ARG;
  if (prefix_len % page_size) return PKV_ERR_UNSUPPORTED;
  if (dtype != PKV_BF16 || head_dim != 128 || page_size != 16) return PKV_ERR_UNSUPPORTED;
  if (!decode_supported(dtype, head_dim, page_size, n_qo_heads / n_kv_heads))
    return PKV_ERR_UNSUPPORTED;
  const size_t need = attn_cascade_workspace_size(n_requests, prefix_len, max_suffix_blocks,
                                                  n_qo_heads, n_kv_heads, head_dim, page_size);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_WORKSPACE;
  CascadeArgs a{};
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.prefix_table = prefix_block_table;
  a.prefix_len = prefix_len;
  a.suffix_table = suffix_block_table;
  a.suffix_lens = suffix_lens;
  a.out = out;
  a.lse = lse;
  a.n_requests = n_requests;
  a.max_suffix_blocks = max_suffix_blocks;
  a.num_pages = num_pages;
  a.n_qo_heads = n_qo_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = head_dim;
  a.page_size = page_size;
  a.scale = scale;
  a.dtype = dtype;
  a.err_flag = err_flag;
  const size_t rows = (size_t)n_requests * n_qo_heads;
  a.prefix_chunks = cascade_prefix_chunks(prefix_len, page_size, n_requests, n_qo_heads, n_kv_heads);
  const SplitPlan suf = cascade_suffix_plan(n_requests, max_suffix_blocks, n_qo_heads, n_kv_heads,
                                            head_dim, PKV_BF16);
  a.suffix_splits = suf.num_splits;
  a.suffix_pages_per_split = suf.pages_per_split;
  char* w = static_cast<char*>(workspace);
  a.pre_o = reinterpret_cast<float*>(w);
  w += align_up((size_t)a.prefix_chunks * rows * head_dim * 4, 256);
  a.pre_lse = reinterpret_cast<float*>(w);
  w += align_up((size_t)a.prefix_chunks * rows * 4, 256);
  a.suf_o = reinterpret_cast<float*>(w);
  w += align_up(rows * suf.num_splits * head_dim * 4, 256);
  a.suf_lse = reinterpret_cast<float*>(w);
  return launch_cascade(a, static_cast<cudaStream_t>(stream));
}

int attn_debug_decode_stall(int page, unsigned long long wait_limit_ns) {
  if (page < -1 || wait_limit_ns > 10000000000ull) return PKV_ERR_INVALID_ARG;
  g_stall_page.store(page, std::memory_order_relaxed);
  g_stall_limit_ns.store(page < 0 ? 0 : (uint64_t)wait_limit_ns, std::memory_order_relaxed);
  return PKV_OK;
}

int attn_flat_gemm_num_splits(int m, int n, int k) {
  if (m < 1 || n < 1 || k < 1) return PKV_ERR_INVALID_ARG;
  if (m > kFlatGemmMaxM) return PKV_ERR_UNSUPPORTED;
  return plan_flat_gemm(m, n, k).splits;
}

int attn_flat_gemm(const void* x, const void* w, void* y, int m, int n, int k, int dtype,
                   int32_t* err_flag, void* stream) {
  const pkv::CallRange range("attn_flat_gemm");
  if (m < 0 || n < 0 || k < 1) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_F32 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return PKV_OK;
  if (!x || !w || !y) return PKV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w)) return PKV_ERR_INVALID_ARG;
  if (dtype != PKV_BF16 || m > kFlatGemmMaxM || k % 8) return PKV_ERR_UNSUPPORTED;
  FlatGemmArgs a{x, w, y, err_flag, m, n, k};
  return launch_flat_gemm(a, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
