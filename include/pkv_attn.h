/*
 * pkv_attn.h: C ABI of the GB300 (sm_103a) paged / causal attention library.
 *
 * Every call computes scaled-dot-product attention, softmax(Q K^T * scale) V
 * ("FlashInfer内核库：利用CUDA Warp-Level Primitives加速级联推理的Attention计算",
 * section 1). The score matrix is never written to memory: scores, softmax and
 * the weighted sum of V stay on chip ("快速注意力内核与算子融合", Q&A on
 * FlashAttention; the FMHA page "TensorRT-LLM深度优化", section 2).
 *
 * Conventions common to every call
 * --------------------------------
 * - Pointers named q, k*, v*, out*, lse*, block_table*, kv_lens*, *_lens,
 *   workspace and err_flag are DEVICE pointers. The caller owns them. The
 *   library never allocates or frees device memory, copies to the host or
 *   synchronises (attn_decode_cascade keeps one side stream and two events per
 *   device, created on first use).
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *   stream. All work is enqueued on it asynchronously. Outputs are valid once
 *   the caller has synchronised with that stream.
 * - Element types: PKV_F32 (float) or PKV_BF16 (bfloat16). Softmax statistics
 *   and partial states are always fp32. Outputs are rounded to the input type
 *   with round-to-nearest-even.
 * - lse is the natural logarithm of sum_j exp(scale * q . k_j), in fp32. It is
 *   -inf when there is no key; the output row is then 0.
 * - GQA: query head h reads KV head h / (n_qo_heads / n_kv_heads).
 *   n_qo_heads must be a multiple of n_kv_heads.
 * - Return value: PKV_OK (0) or a negative PKV_ERR_* code. A non-zero code
 *   means nothing was enqueued, except PKV_ERR_LAUNCH, which reports the CUDA
 *   launch error. Arguments are checked on the host before any launch. No call
 *   aborts the process.
 * - Every compute call runs inside an NVTX range named after it (for example
 *   "attn_decode_paged"), so that Nsight Systems or `ncu --nvtx` can attribute
 *   kernels to calls; without a tool attached a range costs a pointer test.
 * - err_flag (nullable, int32 in device memory) collects problems that only
 *   the device can see, as a bitwise OR of PKV_DEVERR_* bits: a block-table
 *   entry outside [0, num_pages), a length above the table's capacity, or a
 *   pipeline wait that timed out. The rows affected are written as NaN. The
 *   caller clears the flag; the library only ORs bits into it.
 *
 * Paged KV layout
 * ---------------
 *   k_pages, v_pages : [num_pages][n_kv_heads][page_size][head_dim]
 *   block_table      : int32 [batch][max_blocks_per_seq], row-major
 *   kv_lens          : int32 [batch]
 * Token t of sequence b lives in physical page block_table[b][t / page_size],
 * slot t % page_size ("快速注意力内核与算子融合", Q&A on paged attention: a block
 * table maps logical blocks to physical blocks). Table entries at or past
 * ceil(kv_len / page_size), and the slots of the last page past kv_len, are
 * never read.
 */
#ifndef PKV_ATTN_H
#define PKV_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
#define PKV_F32 0
#define PKV_BF16 1
#define PKV_FP8_E4M3 2 /* page pools of attn_decode_paged_fp8 (planning and workspace queries) */

/* status codes */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1) /* null pointer, negative size, inconsistent shape */
#define PKV_ERR_UNSUPPORTED (-2) /* valid but not built: head_dim, page_size, group size, dtype */
#define PKV_ERR_WORKSPACE (-3)   /* workspace missing or smaller than the *_workspace_size call says */
#define PKV_ERR_LAUNCH (-4)      /* a CUDA launch or attribute call failed */
#define PKV_ERR_DEVICE (-5)      /* no usable sm_100-family device is current */

/* device-side error bits ORed into *err_flag */
#define PKV_DEVERR_BAD_PAGE 1 /* a block-table entry outside [0, num_pages) */
#define PKV_DEVERR_BAD_LEN 2  /* a length < 0 or > max_blocks * page_size */
#define PKV_DEVERR_TIMEOUT 4  /* a bounded pipeline wait gave up (nothing hung) */

/* Support set of this build (others return PKV_ERR_UNSUPPORTED):
 *   decode / cascade : head_dim 64 or 128; page_size 16; group size 1, 2, 4 or 8;
 *                      PKV_F32 or PKV_BF16 (cascade: PKV_BF16, head_dim 128)
 *   prefill          : head_dim 128; PKV_BF16; any seq_len >= 1
 *   flat GEMM        : PKV_BF16; 1 <= m <= 64; k a multiple of 8
 */

/* Human-readable name of a status code. Static storage; never NULL. */
const char* attn_status_string(int status);

/* Text of the CUDA error behind the most recent PKV_ERR_LAUNCH returned on the
 * calling host thread ("no error" if there was none). Static storage; never NULL.
 * A diagnostic for callers; the pages define no counterpart. */
const char* attn_last_cuda_error_string(void);

/*
 * Number of KV splits the decode calls use for this shape and dtype. num_splits > 0
 * is taken as asked (capped at max_blocks_per_seq); 0 lets the library choose from
 * the shape, the SM count of the current device and how many decode CTAs fit on an
 * SM, as the split count that minimises (waves of CTAs) x (pages per CTA + 4), plus 24
 * for the split merge when there is more than one split (so small problems get one
 * split and no merge launch). A split covers a contiguous range of
 * ceil(max_blocks_per_seq / splits) pages of a sequence.
 * FlashDecoding computes each partial softmax independently and combines them
 * all at the end ("【FlashAttention-V4，非官方】FlashDecoding++", section 1).
 * Returns the split count (>= 1) or a negative PKV_ERR_* code.
 */
int attn_decode_num_splits(int batch, int max_blocks_per_seq, int n_qo_heads, int n_kv_heads,
                           int head_dim, int page_size, int num_splits, int dtype);

/*
 * Workspace bytes attn_decode_paged and attn_decode_paged_unified_max need for
 * this shape: the fp32 partial states O[batch][n_qo_heads][splits][head_dim] and
 * LSE[batch][n_qo_heads][splits]. It is 0 when one split suffices. Returns
 * (size_t)-1 for invalid arguments.
 */
size_t attn_decode_workspace_size(int batch, int max_blocks_per_seq, int n_qo_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_splits,
                                  int dtype);

/*
 * Single-token decode over a paged KV cache.
 *
 *   q     : [batch][n_qo_heads][head_dim], dtype
 *   out   : [batch][n_qo_heads][head_dim], dtype (must not alias an input)
 *   lse   : [batch][n_qo_heads] fp32 (nullable: not written)
 *   scale : multiplies q . k before the softmax (1/sqrt(head_dim) for the
 *           textbook form)
 *
 * The pages read K and V through a block table that maps a sequence's logical
 * blocks to physical pages ("快速注意力内核与算子融合", Q&A on paged attention), and
 * split the keys into partial softmax states that are combined at the end
 * ("【FlashAttention-V4，非官方】FlashDecoding++", section 1, on FlashDecoding).
 * One unit of work is (sequence, KV head, split): that split's K/V pages are
 * streamed through the block table into a shared-memory ring, with a running max
 * and sum (online softmax), and a partial (O, LSE) state is written. A merge kernel
 * (one CTA per output row, launched on `stream` as a programmatic dependent of the
 * decode so that it is placed while the decode's last CTAs run) then combines the
 * partials by log-sum-exp. Sequences whose pages fit in one split are written directly. With 1 or 2 query heads per KV head (and for fp32) the dot
 * products and sums run on the CUDA cores, one CTA per unit, the group's queries in
 * registers. For bf16, head_dim 128 and 4 or 8 query heads per KV head they run on
 * the tcgen05 tensor cores: 128-key tiles (8 pages) against the group's queries,
 * padded to 16, with fp32 accumulators in tensor memory; CTAs take units from the
 * grid until none is left, and with one split per sequence (batch <= 2048) the longest
 * sequences' units are handed out first. The workspace (device, >= attn_decode_workspace_size bytes,
 * 256-byte aligned) holds the partials; its contents on entry do not matter.
 */
int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* block_table, const int32_t* kv_lens, void* out, float* lse,
                      int batch, int max_blocks_per_seq, int num_pages, int n_qo_heads,
                      int n_kv_heads, int head_dim, int page_size, float scale, int num_splits,
                      int dtype, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                      void* stream);

/*
 * Allocation-free variant of attn_decode_paged (the pages have no counterpart;
 * this is a convenience of the library).
 *
 * Some callers cannot allocate device memory when they call in. Examples are an
 * inference runtime's plugin or enqueue hook that is not allowed to allocate
 * while it runs, and a process that reserved all device memory up front for its
 * own pool. Those callers cannot supply the workspace that attn_decode_paged
 * wants. This entry point keeps the split partial states in a scratch array
 * that the library owns instead: PKV_NOALLOC_SCRATCH_BYTES bytes of static
 * device memory, held on every GPU that loads the library until the process
 * exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - Arguments, layouts and results are those of attn_decode_paged, minus the
 *   workspace. The output equals attn_decode_paged's for the same split count.
 * - Returns PKV_ERR_WORKSPACE when the shape needs more than
 *   PKV_NOALLOC_SCRATCH_BYTES of partial states, i.e. when
 *   attn_decode_workspace_size(...) > PKV_NOALLOC_SCRATCH_BYTES. Fewer splits
 *   (num_splits) or a smaller batch fit.
 * - The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress) with that device current, and caches it with the
 *   unique id of the current context (cuCtxGetId). Make that first call before
 *   any stream capture on that device. cudaDeviceReset destroys the array with
 *   the device's context; the first call in the context that replaces it sees
 *   another context id and looks the address up again (again outside a
 *   capture). Where the driver gives no context id, every call looks it up.
 * - Every call on a device shares the one array. Calls whose kernels overlap on
 *   the GPU (different streams, no ordering between them) race on it and give
 *   wrong results; order them, e.g. on one stream. The array keeps the last
 *   call's contents. Nothing in it needs to start at zero: every partial state
 *   that a call reads was written by the same call.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB of fp32 partial states */

int attn_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* kv_lens, void* out,
                              float* lse, int batch, int max_blocks_per_seq, int num_pages,
                              int n_qo_heads, int n_kv_heads, int head_dim, int page_size,
                              float scale, int num_splits, int dtype, int32_t* err_flag,
                              void* stream);

/*
 * Decode with FlashDecoding++'s asynchronised softmax with a unified maximum
 * value ("【FlashAttention-V4，非官方】FlashDecoding++", sections 1 and 3).
 * Scaled logits are exponentiated against the preset value `phi` (natural-log
 * units, same units as lse), not against a running maximum. There is no per-tile
 * max synchronisation, and partial states that share phi add up without
 * rescaling. The pages leave the bound and the fallback open. This library's
 * reading:
 *   - when a tile holds a logit above phi + 60, the CTA raises its reference
 *     value to that tile's max and rescales what it has accumulated;
 *   - when a tile lies wholly below phi - 60 before anything was accumulated,
 *     the reference value drops to the tile's max.
 * Either event adds 1 to *fallback_count (nullable, int32 device counter,
 * caller-cleared). The result equals attn_decode_paged up to rounding. Arguments,
 * workspace and errors are as for attn_decode_paged.
 */
int attn_decode_paged_unified_max(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* kv_lens, void* out,
                                  float* lse, int batch, int max_blocks_per_seq, int num_pages,
                                  int n_qo_heads, int n_kv_heads, int head_dim, int page_size,
                                  float scale, int num_splits, int dtype, float phi,
                                  int32_t* fallback_count, void* workspace,
                                  size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * Decode over FP8 page pools. FP8 cuts attention's memory traffic ("TensorRT-LLM
 * 深度优化：利用FMHA（Fused Multi-Head Attention）内核加速Hopper架构推理", section 4);
 * the page names neither a format nor a scaling, and this library's reading is:
 *   - k_pages, v_pages hold E4M3 codes (the OCP 8-bit floating-point format: bias 7,
 *     3 mantissa bits, no infinities), one byte per element, in the paged layout;
 *   - k_scale, v_scale : fp32 [num_pages][n_kv_heads], one scale per (page, KV head)
 *     tile; an element's value is e4m3(code) * scale;
 *   - q and out are bf16 (dtype PKV_BF16 implied); lse, workspace, splits and
 *     err_flag are as for attn_decode_paged, with the workspace size from
 *     attn_decode_workspace_size(..., PKV_FP8_E4M3).
 * The result is the attention of attn_decode_paged over the dequantised values, with
 * the per-tile scales applied to the dot products and to the softmax weights.
 * Arithmetic: codes become f16 exactly; q is scaled per head by a power of two that
 * brings its largest magnitude to [2^14, 2^15) and converted to f16 (exact for bf16 q,
 * whatever its range, except for elements more than 2^24 below the head's largest);
 * dot products and the weighted sums of V accumulate in fp32. A softmax weight times the
 * tile's V scale enters the V sum as an f16 value (11-bit significand, normal from 2^-14
 * to 65504): V scales above 65504 are not supported, and below about 2^-14 such a weight
 * keeps an absolute precision of 2^-24. Pools
 * must be 16-byte aligned, and n_kv_heads must be even (the CUDA-core kernel's CTA takes two
 * adjacent KV heads). Built for head_dim 64 and 128, page_size 16 and GQA groups 1, 2, 4 and
 * 8; other shapes return PKV_ERR_UNSUPPORTED. At head_dim 128 with 4 or 8 query heads per KV
 * head the products run on the tcgen05 tensor cores: converter warps take each tile's codes
 * to f16 in shared memory (exactly), q goes to f16 as above, the K scale multiplies each
 * logit and a weight times its page's V scale enters the V product as f16, with fp32
 * accumulation; the other shapes run on the CUDA cores.
 */
int attn_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages,
                          const float* k_scale, const float* v_scale, const int32_t* block_table,
                          const int32_t* kv_lens, void* out, float* lse, int batch,
                          int max_blocks_per_seq, int num_pages, int n_qo_heads, int n_kv_heads,
                          int head_dim, int page_size, float scale, int num_splits,
                          void* workspace, size_t workspace_bytes, int32_t* err_flag,
                          void* stream);

/*
 * Chunked prefill over the paged cache: each sequence b already holds prefix_lens[b]
 * tokens and appends chunk_len new ones, whose K and V the caller has already written
 * into the pages at positions prefix_lens[b] .. prefix_lens[b] + chunk_len - 1. New
 * token i attends to keys 0 .. prefix_lens[b] + i of its own sequence (the causal mask
 * with an offset), read through the block table ("快速注意力内核与算子融合", Q&A on
 * paged attention and on FlashAttention; the pages do not describe the combination).
 *
 *   q, out      : bf16 [batch][chunk_len][n_qo_heads][head_dim], contiguous
 *   k_pages, v_pages, block_table : the paged layout above (bf16 pools)
 *   prefix_lens : int32 [batch]; prefix_lens[b] + chunk_len must fit the table's
 *                 max_blocks_per_seq pages (else PKV_DEVERR_BAD_LEN, computed on a
 *                 clamped length)
 *   lse         : fp32 [batch][n_qo_heads][chunk_len] (nullable)
 * Both products run on the tcgen05 tensor cores (the prefill kernel's paged mode). Built
 * for bf16, head_dim 128, page_size 16 and GQA groups dividing 128; all pointers 16-byte
 * aligned.
 */
int attn_prefill_paged_chunk(const void* q, const void* k_pages, const void* v_pages,
                             const int32_t* block_table, const int32_t* prefix_lens, void* out,
                             float* lse, int batch, int chunk_len, int max_blocks_per_seq,
                             int num_pages, int n_qo_heads, int n_kv_heads, int head_dim,
                             int page_size, float scale, int dtype, int32_t* err_flag,
                             void* stream);

/*
 * Merge two partial softmax states over disjoint key sets into one
 * ("【FlashAttention-V4，非官方】FlashDecoding++", section 1: partial softmax
 * results are updated at the end):
 *   M = max(lse_a, lse_b), w_x = exp(lse_x - M),
 *   out = (w_a out_a + w_b out_b) / (w_a + w_b), lse = M + ln(w_a + w_b).
 * Two -inf sides give out = 0, lse = -inf.
 *
 *   out_a, out_b : fp32 [n_rows][head_dim];  lse_a, lse_b : fp32 [n_rows]
 *   out          : out_dtype [n_rows][head_dim]; with out_dtype PKV_F32 it may
 *                  alias out_a or out_b exactly
 *   lse          : fp32 [n_rows] (nullable); may alias lse_a or lse_b exactly
 * n_rows is every leading dimension flattened (e.g. batch * heads).
 */
int attn_merge_states(const float* out_a, const float* lse_a, const float* out_b,
                      const float* lse_b, void* out, float* lse, int n_rows, int head_dim,
                      int out_dtype, void* stream);

/*
 * Causal self-attention for prefill: query i of a sequence attends to keys
 * 0..i of the same sequence. The query length equals the key length.
 *
 *   q, out : [batch][seq_len][n_qo_heads][head_dim], dtype, contiguous
 *   k, v   : [batch][seq_len][n_kv_heads][head_dim], dtype, contiguous
 *   lse    : fp32 [batch][n_qo_heads][seq_len] (nullable)
 *
 * The work is tiled as in FlashAttention: per tile, compute the scores,
 * update the softmax statistics and accumulate the output on chip, so the
 * T x T score matrix never reaches HBM ("快速注意力内核与算子融合", Q&A on
 * FlashAttention). Both products run on the tcgen05 tensor cores with fp32
 * accumulators in tensor memory, fed by TMA. All pointers must be 16-byte
 * aligned.
 */
int attn_prefill_causal(const void* q, const void* k, const void* v, void* out, float* lse,
                        int batch, int seq_len, int n_qo_heads, int n_kv_heads, int head_dim,
                        float scale, int dtype, int32_t* err_flag, void* stream);

/* Workspace bytes attn_decode_cascade needs (fp32 partial states). (size_t)-1 on bad args. */
size_t attn_cascade_workspace_size(int n_requests, int prefix_len, int max_suffix_blocks,
                                   int n_qo_heads, int n_kv_heads, int head_dim, int page_size);

/*
 * Cascade (shared-prefix) decode. Every request's sequence is one shared prefix,
 * whose pages are listed once in prefix_block_table, followed by that request's
 * own suffix pages. Two readings meet here: "级联推理", which splits attention
 * into stages that each handle part of the data (FlashInfer page, sections 2
 * and 4), and prefix sharing in the paged cache ("快速注意力内核与算子融合", Q&A
 * on paged attention). The prefix is attended once per KV head for the queries
 * of all requests and that KV head's query heads, as one tensor-core product.
 * The suffix is attended per request. The two partial states are merged by
 * log-sum-exp.
 *
 *   q, out             : [n_requests][n_qo_heads][head_dim], dtype
 *   lse                : fp32 [n_requests][n_qo_heads] (nullable)
 *   prefix_block_table : int32 [ceil(prefix_len / page_size)]
 *   suffix_block_table : int32 [n_requests][max_suffix_blocks]
 *   suffix_lens        : int32 [n_requests] (0 allowed)
 *   workspace          : >= attn_cascade_workspace_size bytes, 256-byte aligned
 * The result equals attn_decode_paged over the concatenated sequences, up to
 * rounding.
 *
 * With 4 or 8 query heads per KV head (bf16, head_dim 128) the suffix runs on the
 * tensor-core decode, one unit per (request, KV head), launched on `stream` right after
 * the prefix product so that it starts while the prefix product finishes (programmatic
 * dependent launch); each unit waits for the prefix grid only before it merges the
 * prefix's partial states with its own and writes the request's rows. Other groups run
 * the prefix product on a side stream of the library's (one per device, created with two
 * events on first use and kept for the life of the process), forked from and joined back
 * into `stream` with events, so that it overlaps the CUDA-core suffix decode, and a merge
 * kernel combines the states. Either way the call completes in `stream` order and may be
 * captured.
 */
int attn_decode_cascade(const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* prefix_block_table, int prefix_len,
                        const int32_t* suffix_block_table, const int32_t* suffix_lens, void* out,
                        float* lse, int n_requests, int max_suffix_blocks, int num_pages,
                        int n_qo_heads, int n_kv_heads, int head_dim, int page_size, float scale,
                        int dtype, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                        void* stream);

/*
 * Flat GEMM of the decode phase: y = x w^T for a few tokens ("【FlashAttention-V4，非官方】
 * FlashDecoding++", section 4, Flat GEMM Optimization with Double Buffering; the problem is
 * stated in sections 1 and 2). In decode the projections either side of attention see only
 * a few tokens at a time, so the GEMM is flat (with one token, a GEMV); the page pads the
 * token dimension with zeros to 8 instead of the libraries' 64 and overlaps the loads of
 * the next tile with the products of the current one with two shared-memory buffers.
 *
 *   x : bf16 [m][k], the m tokens, row-major
 *   w : bf16 [n][k], the k x n weight operand passed transposed (each of its n columns
 *       contiguous, as projection weights are stored)
 *   y : bf16 [m][n] = x w^T, fp32 accumulation, rounded to nearest even; must not alias
 *       x or w
 * Built for dtype PKV_BF16, 1 <= m <= 64, k >= 1 a multiple of 8 (16-byte rows), any n;
 * x and w 16-byte aligned. m = 0 or n = 0 does nothing. Other shapes return
 * PKV_ERR_UNSUPPORTED. err_flag (nullable) gets PKV_DEVERR_TIMEOUT if a bounded wait gave
 * up; the 128 columns of y that CTA group owns are then NaN.
 *
 * The weights stream through the tcgen05 tensor cores 128 rows at a time (the product's M
 * dimension); the tokens are the product's N dimension, padded with zeros to 16, 32 or 64
 * by the TMA loads (16 is the narrowest product with 128 rows). A ring of shared-memory
 * stages, fed by TMA, overlaps the loads of the next 64-column slice of K with the
 * products of the current one (the page's double buffering, with more than two buffers).
 * K is split over a thread-block cluster of up to 8 CTAs, whose partial tiles are summed
 * through distributed shared memory: one launch, and no workspace.
 */
int attn_flat_gemm(const void* x, const void* w, void* y, int m, int n, int k, int dtype,
                   int32_t* err_flag, void* stream);

/*
 * Failure-handling hook for tests (the pages have no counterpart). It lets a test make a
 * bounded wait inside the decode kernel run out, without faulting or hanging anything:
 * after attn_debug_decode_stall(page, wait_limit_ns) with page >= 0, every launch of
 * attn_decode_paged, attn_decode_paged_unified_max, attn_decode_paged_fp8 and
 * attn_decode_paged_noalloc in this process has the producer warp of each CTA withhold
 * the copies of the page-th page of its split (on the tensor-core path: the K copies of
 * the 128-key tile that holds it) and the arrival that would announce them, and every
 * pipeline wait of those launches gives up after wait_limit_ns nanoseconds (0 keeps the
 * default of 2 s). The consumer waiting for that page then times out: the kernel ORs
 * PKV_DEVERR_TIMEOUT into err_flag, waits (within the same limit) for the copies it did
 * issue, writes the rows (or split partials) of the unit it was working on, and of any
 * later unit it had taken, as NaN and returns, so the context stays usable. attn_debug_decode_stall(-1, 0) turns it off. Not for use
 * beside production calls: the setting is process-wide. Returns PKV_OK, or
 * PKV_ERR_INVALID_ARG for page < -1 or a limit above 10 s.
 */
int attn_debug_decode_stall(int page, unsigned long long wait_limit_ns);

/* How many CTAs (the cluster size, 1..8) share K for this shape on the current device;
 * a negative PKV_ERR_* code for shapes attn_flat_gemm rejects. */
int attn_flat_gemm_num_splits(int m, int n, int k);

#ifdef __cplusplus
}
#endif

#endif /* PKV_ATTN_H */
