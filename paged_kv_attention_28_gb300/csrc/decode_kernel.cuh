// Paged single-token decode kernel (sm_103a).
//
// One CTA per (KV split, KV head, sequence); the FP8 variant's CTA takes two adjacent
// KV heads (see DecodeCfg). A producer warp streams the
// split's (page, KV head) tiles of K and V (page_size x head_dim contiguous
// elements each) through the block table into a ring of shared-memory stages.
// It uses one-dimensional bulk TMA copies that complete on an mbarrier.
// Consumer warps take the pages in turn. Each keeps the query heads of its GQA
// group in registers and reduces the q.k dot products and the running
// max/sum with __shfl_xor_sync. The block-table mapping is from
// "快速注意力内核与算子融合" (Q&A on paged attention); the warp-shuffle
// reductions are the warp-level primitives of the FlashInfer page (section 3).
//
// Softmax statistics are carried in base-2 units: logits are prescaled by
// scale*log2(e), exponentials are ex2, and lse = (ref + log2 l) * ln 2.
//
// Two ways to pick the reference value that logits are exponentiated against:
//  * online (FlashAttention/FlashDecoding): the running max. When a chunk
//    raises it, the accumulated sum and output are rescaled.
//  * unified (FlashDecoding++ asynchronised softmax, "【FlashAttention-V4，
//    非官方】FlashDecoding++" sections 1 and 3): a preset phi shared by every
//    partial, with no max tracking. A warp moves off phi only when a chunk
//    would overflow (a logit above phi + beta) or, for its first chunk, would
//    underflow entirely (every logit below phi - beta). Each such event is
//    counted.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Unified-max safety margin in natural-log units: exp(60) * 2^20 terms stays
// far below FLT_MAX, and a chunk 60 below the reference contributes < e^-60.
constexpr float kUnifiedBeta = 60.0f;

// Lanes per token row: 16 halves the registers a lane holds for G >= 4 (q and the
// accumulators of G heads), so that G = 4 fits three CTAs per SM, the online and the
// unified-max variant alike (with the reduce-scatter below, 8 lanes and two CTAs per SM
// measured 5 % slower on the unified-max variant and 5 % slower on the online one).
// FP8: the page pools hold E4M3 codes with one float scale per (page, KV head) tile of K
// and of V; q and the output stay T (bf16). A stage then carries half the bytes and the
// CTA half the shared memory. A CTA takes two adjacent KV heads so that each bulk copy
// still moves 4 KiB (both heads' tiles of a page); with 2 KiB copies the batch ran at half
// the DRAM throughput. G = 1 runs six CTAs per SM. Measured on the Llama-7B batch: one head
// per CTA with 3, 5, 6, 7 CTAs per SM 130, 102, 93, 106 us; two heads per CTA 77 us.
template <typename T, int D, int P, int G, bool UNIFIED = false, bool FP8 = false>
struct DecodeCfg {
  using KV = std::conditional_t<FP8, uint8_t, T>;  // element type of the page pools
  static constexpr int ES = sizeof(KV);
  static constexpr int LPT = (G >= 4) ? 16 : 8;
  static constexpr int TPI = 32 / LPT;             // token rows a warp covers per step
  static constexpr int DPL = D / LPT;              // head dims held per lane
  static constexpr int VEC = (16 / ES < DPL) ? 16 / ES : DPL;  // elements per smem load
  static constexpr int NV = DPL / VEC;             // loads per row per lane
  static constexpr int ITERS = P / TPI;            // steps per page
  static constexpr int NIT_MAX = (32 / G) > 0 ? (32 / G) : 1;
  static constexpr int NIT = ITERS < NIT_MAX ? ITERS : NIT_MAX;  // steps per softmax chunk
  static constexpr int NCHUNK = ITERS / NIT;
  static constexpr int TILE = P * D * ES;          // bytes of one (page, KV head) tile
  // FP8: a CTA takes two adjacent KV heads, so one bulk copy moves both heads' tiles of a
  // page (2 x 2 KiB, contiguous in the pool) instead of two copies of 2 KiB.
  static constexpr int HPC = FP8 ? 2 : 1;          // KV heads per CTA
  static constexpr int STAGE = HPC * TILE;         // bytes of K (or V) in one ring stage
  static constexpr int NW = 4;                     // consumer warps
  static constexpr int WPH = NW / HPC;             // consumer warps per KV head
  // bf16 with one query head per KV head: a 4-stage ring and five CTAs per SM keep more
  // pages in flight per SM than 8 stages and three CTAs (measured 6359 against 6259 GB/s
  // on the Llama-7B batch; 4 stages and four CTAs 6012). fp32 at head_dim 64 with one query
  // head per KV head (4 KiB tiles, few CTAs): 16 stages, so that a 256-token sequence's
  // pages are all requested at once (32 such calls back to back: 194 against 206 us).
  static constexpr int NSTAGE =
      (G == 1 && sizeof(T) == 2) ? 4 : (G == 1 && sizeof(T) == 4 && D == 64 && !FP8) ? 16 : 8;  // multiple of NW
  static constexpr int THREADS = (NW + 1) * 32;
  // G = 8 (fp32, head_dim 64 and FP8: the bf16 head_dim-128 groups of 4 and 8 run on the
  // tensor cores) asks for no occupancy, and fp32 G = 4 at head_dim 128 for two CTAs per
  // SM, so that q and the accumulators stay in registers instead of spilling.
  static constexpr int MIN_BLOCKS = G >= 8 ? 1 : (G >= 4 && sizeof(T) == 4 && D >= 128) ? 2 : G > 1 ? 3 : FP8 ? 6 : sizeof(T) == 2 ? 5 : 3;
  // G >= 4: the row's lanes reduce the G dot products by halving exchanges, after which
  // each lane holds one head's full score (reduce_scatter_heads).
  static constexpr bool SCATTER = G >= 4 && G <= LPT;
  static constexpr int BAR_OFF = 2 * NSTAGE * STAGE;
  static constexpr int FLAG_OFF = BAR_OFF + 2 * NSTAGE * 8;
  static constexpr int SCALE_OFF = FLAG_OFF + 16;  // FP8: (k_scale, v_scale) of each stage
  static constexpr int SMEM = SCALE_OFF + (FP8 ? NSTAGE * HPC * 8 : 0);
  static_assert(D % LPT == 0 && DPL % VEC == 0 && VEC % 2 == 0, "head_dim split");
  static_assert(P % TPI == 0 && ITERS % NIT == 0, "page split");
  static_assert(NSTAGE % NW == 0, "stage ownership");
  static_assert(TILE % 16 == 0, "bulk copy granularity");
  static_assert(NW * G * (D + 2) * 4 <= 2 * NSTAGE * STAGE, "combine scratch fits in the ring");
  static_assert(NW % HPC == 0 && NSTAGE % WPH == 0, "stage ownership per head");
};

__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// Two independent fp32 fused multiply-adds in one instruction (sm_100 family).
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Reduces G per-lane partial dot products over the LPT lanes of a token row so that
// each lane ends with the full sum of one head: head j / (LPT / G), j = lane % LPT.
// Stage r exchanges half of the values still held with the lane LPT >> (r + 1) away:
// the lane with that bit set keeps the upper half of the heads, its partner the lower.
// After log2 G stages one value is left, summed over the lanes that differ in those
// bits, and plain xor steps sum it over the remaining ones. That is G - 1 + log2(LPT/G)
// shuffles per row where reducing every head over every lane takes G * log2 LPT.
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter_heads(const float (&v)[G], int j) {
  float cur[G];
#pragma unroll
  for (int k = 0; k < G; ++k) cur[k] = v[k];
#pragma unroll
  for (int half = G / 2, off = LPT / 2; half >= 1; half /= 2, off /= 2) {
    const bool up = (j & off) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float keep = up ? cur[k + half] : cur[k];
      const float send = up ? cur[k] : cur[k + half];
      cur[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float x = cur[0];
#pragma unroll
  for (int off = LPT / (2 * G); off >= 1; off /= 2) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// v[h] for a per-lane head index h (selects, no local-memory indexing).
template <int G>
__device__ __forceinline__ float pick(const float (&v)[G], int h) {
  float x = v[0];
#pragma unroll
  for (int k = 1; k < G; ++k) x = (h == k) ? v[k] : x;
  return x;
}

struct DecodeFlags {
  int abort_;
  int bad_page;
  int issued;
  int fallbacks;
};

// Loads VEC elements of one K or V row from shared memory (VEC * sizeof(T)
// bytes, aligned) as VEC/2 packed (even, odd) fp32 pairs. bf16 -> fp32 is a
// 16-bit left shift of the bit pattern.
// FP8 rows stay in f16: two E4M3 codes (element 2i in the low byte) convert exactly to an
// f16 pair in one instruction, and the dot products and the PV sums take f16 operands
// with fp32 accumulation (mixed-precision fma), so no code is widened to fp32 on its own.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t pair) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(pair & 0xffffu)));
  return r;
}

// VEC E4M3 codes from shared memory as VEC/2 f16 pairs.
template <int VEC>
__device__ __forceinline__ void load_row_h2(const uint8_t* p, uint32_t* h2) {
  static_assert(VEC == 4 || VEC == 8 || VEC == 16, "E4M3 rows are read 4, 8 or 16 codes at a time");
  if constexpr (VEC == 4) {
    const uint32_t x = *reinterpret_cast<const uint32_t*>(p);
    h2[0] = e4m3x2_to_h2(x);
    h2[1] = e4m3x2_to_h2(x >> 16);
  } else if constexpr (VEC == 8) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    h2[0] = e4m3x2_to_h2(x.x);
    h2[1] = e4m3x2_to_h2(x.x >> 16);
    h2[2] = e4m3x2_to_h2(x.y);
    h2[3] = e4m3x2_to_h2(x.y >> 16);
  } else {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h2[2 * i] = e4m3x2_to_h2(w[i]);
      h2[2 * i + 1] = e4m3x2_to_h2(w[i] >> 16);
    }
  }
}

// lo += a.lo * b.lo, hi += a.hi * b.hi: f16 pairs in, fp32 sums.
__device__ __forceinline__ void fma_h2_f32(uint32_t a, uint32_t b, float& lo, float& hi) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}

// The fp32 pair acc += (v.lo, v.hi) * p for an f16 pair v and an f16 scalar p.
__device__ __forceinline__ uint64_t fma_h2s_f32x2(uint32_t v, unsigned short p, uint64_t acc) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc));
  asm("{\n\t.reg .b16 vl, vh;\n\tmov.b32 {vl, vh}, %2;\n\t"
      "fma.rn.f32.f16 %0, vl, %3, %0;\n\tfma.rn.f32.f16 %1, vh, %3, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(v), "h"(p));
  return pk2(lo, hi);
}

__device__ __forceinline__ unsigned short f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

template <typename T, int VEC>
__device__ __forceinline__ void load_row_pairs(const T* p, uint64_t* f2) {
  if constexpr (sizeof(T) == 4) {
    if constexpr (VEC == 4) {
      const float4 x = *reinterpret_cast<const float4*>(p);
      f2[0] = pk2(x.x, x.y);
      f2[1] = pk2(x.z, x.w);
    } else {
      const float2 x = *reinterpret_cast<const float2*>(p);
      f2[0] = pk2(x.x, x.y);
    }
  } else {
    if constexpr (VEC == 8) {
      const uint4 x = *reinterpret_cast<const uint4*>(p);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) f2[i] = pk2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    } else {
      const uint2 x = *reinterpret_cast<const uint2*>(p);
      f2[0] = pk2(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xffff0000u));
      f2[1] = pk2(__uint_as_float(x.y << 16), __uint_as_float(x.y & 0xffff0000u));
    }
  }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Writes the rows of one (sequence, KV head) group: NaN (bad input), or 0 / -inf
// (empty sequence). Used by the split-0 CTA only.
template <typename T, int D, int G>
__device__ void write_group_const(const DecodeArgs& a, int b, int g, float o, float l) {
  T* out = static_cast<T*>(a.out);
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = g * G + idx / D;
    out[((size_t)b * a.n_qo_heads + h) * D + idx % D] = from_f32<T>(o);
    if (a.lse && idx % D == 0) a.lse[(size_t)b * a.n_qo_heads + h] = l;
  }
}

template <typename T, int D, int P, int G, bool UNIFIED, bool FP8 = false>
__global__ void __launch_bounds__(DecodeCfg<T, D, P, G, UNIFIED, FP8>::THREADS,
                                  DecodeCfg<T, D, P, G, UNIFIED, FP8>::MIN_BLOCKS)
decode_paged_kernel(const DecodeArgs a) {
  using C = DecodeCfg<T, D, P, G, UNIFIED, FP8>;
  using KV = typename C::KV;
  extern __shared__ __align__(128) unsigned char smem[];
  const int split = blockIdx.x;
  const int g0 = blockIdx.y * C::HPC;  // first KV head of this CTA
  const int b = blockIdx.z;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int hh = warp < C::NW ? warp / C::WPH : 0;  // a consumer warp's head within the CTA
  const int g = g0 + hh;
  // The split merge, launched next on the same stream, may take its place on the SMs once
  // every CTA of this grid has started; it waits for this grid before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int kv_len = __ldg(a.kv_lens + b);
  // The split's first 32 table entries are requested together with the length (their
  // addresses do not depend on it), so the page copies wait for one round trip, not two.
  // Entries past the sequence's end are read but never used; all lie inside the table.
  int phys_first = 0;
  if (warp == C::NW) {
    const int idx = split * a.pages_per_split + lane;
    if (lane < a.pages_per_split && idx < a.max_blocks)
      phys_first = __ldg(a.block_table + (size_t)b * a.max_blocks + idx);
  }
  if (kv_len < 0 || kv_len > a.max_blocks * P) {
    if (split == 0) {
      if (threadIdx.x == 0) set_err(a.err_flag, PKV_DEVERR_BAD_LEN);
      if (!a.partial_only)
        for (int k = 0; k < C::HPC; ++k) write_group_const<T, D, G>(a, b, g0 + k, NAN, NAN);
    }
    return;
  }
  const int nblk = (kv_len + P - 1) / P;
  const int n_live = (nblk + a.pages_per_split - 1) / a.pages_per_split;
  if (n_live == 0) {
    if (split == 0 && !a.partial_only)
      for (int k = 0; k < C::HPC; ++k) write_group_const<T, D, G>(a, b, g0 + k, 0.0f, -INFINITY);
    return;
  }
  if (split >= n_live) return;
  const int first = split * a.pages_per_split;
  const int n_pages = min(a.pages_per_split, nblk - first);
  const bool final_write = (n_live == 1) && !a.partial_only;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::BAR_OFF;
  const uint32_t bar_empty = bar_full + C::NSTAGE * 8;
  DecodeFlags* flags = reinterpret_cast<DecodeFlags*>(smem + C::FLAG_OFF);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, C::HPC);  // one arrival from each head's consumer
    }
    flags->abort_ = 0;
    flags->bad_page = 0;
    flags->issued = 0;
    flags->fallbacks = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::NW) {
    // ------------------------------------------------------------ producer warp
    const int32_t* trow = a.block_table + (size_t)b * a.max_blocks + first;
    const uint64_t pol = policy_evict_first();
    const char* kbase = static_cast<const char*>(a.k_pages);
    const char* vbase = static_cast<const char*>(a.v_pages);
    bool ok = true;
    int issued = 0;
    for (int base = 0; base < n_pages && ok; base += 32) {
      const int idx = base + lane;
      const int phys = (idx < n_pages) ? (base == 0 ? phys_first : __ldg(trow + idx)) : 0;
      const bool bad = (idx < n_pages) && (phys < 0 || phys >= a.num_pages);
      const unsigned badm = __ballot_sync(0xffffffffu, bad);
      if (badm && lane == 0) {
        set_err(a.err_flag, PKV_DEVERR_BAD_PAGE);
        flags->bad_page = 1;
      }
      const int cnt = min(32, n_pages - base);
      // The whole warp runs the loop (the ring waits are warp-wide) and one elected
      // lane issues each page's copies.
      for (int k = 0; k < cnt; ++k) {
        const int p = __shfl_sync(0xffffffffu, phys, k);
        const int i = base + k;
        const int s = i % C::NSTAGE;
        const int use = i / C::NSTAGE;
        if (use > 0 && !warp_wait(bar_empty + 8 * s, (use - 1) & 1, a.wait_limit_ns)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          if constexpr (FP8) {
            // the stage's scales (per head of the CTA), published by the arrive below
            float* scl = reinterpret_cast<float*>(smem + C::SCALE_OFF) + 2 * C::HPC * s;
            const bool bad_k = (badm >> k) & 1u;
            for (int h2 = 0; h2 < C::HPC; ++h2) {
              const size_t si = (size_t)(bad_k ? 0 : p) * a.n_kv_heads + g0 + h2;
              scl[2 * h2] = bad_k ? 0.0f : __ldg(a.k_scale + si);
              scl[2 * h2 + 1] = bad_k ? 0.0f : __ldg(a.v_scale + si);
            }
          }
          if ((badm >> k) & 1u) {
            mbar_arrive(bar_full + 8 * s);  // completes the phase with no data
          } else if (i == a.stall_page) {
            // injected stall: neither copies nor an arrival, so this stage's consumer
            // waits until its limit runs out
          } else {
            // the CTA's HPC heads' tiles of a page are adjacent in the pool: one copy each
            const size_t off = ((size_t)p * a.n_kv_heads + g0) * C::TILE;
            mbar_arrive_expect_tx(bar_full + 8 * s, 2 * C::STAGE);
            bulk_g2s_hint(sbase + s * C::STAGE, kbase + off, C::STAGE, bar_full + 8 * s, pol);
            bulk_g2s_hint(sbase + (C::NSTAGE + s) * C::STAGE, vbase + off, C::STAGE,
                          bar_full + 8 * s, pol);
          }
        }
        __syncwarp();
        issued = i + 1;
      }
    }
    if (lane == 0) {
      flags->issued = issued;
      if (!ok) {
        flags->abort_ = 1;
        set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
      }
    }
  }

  // ---------------------------------------------------------------- consumer warps
  const int tg = lane / C::LPT;  // token row within a step
  const int j = lane % C::LPT;   // column group within the row
  constexpr int DP2 = C::DPL / 2;  // packed pairs per lane
  float ref[G], lsum[G];
  uint64_t acc2[G][DP2];
#pragma unroll
  for (int gi = 0; gi < G; ++gi) {
    ref[gi] = UNIFIED ? a.phi * kLog2e : -INFINITY;
    lsum[gi] = 0.0f;
#pragma unroll
    for (int e = 0; e < DP2; ++e) acc2[gi][e] = 0ull;  // (+0, +0)
  }
  int fallbacks = 0;
  // SCATTER: this lane's head and its running sum (lsum[] is filled after the loop)
  static_assert(G <= C::LPT, "a token row has at least one lane per head");
  const int h_own = j / (C::LPT / G);
  float lsum_own = 0.0f;

  if (warp < C::NW) {
    // q as fp32 pairs prescaled by scale*log2(e); FP8: f16 pairs, the scale and the tile's
    // k_scale multiply the finished dot product.
    using QP = std::conditional_t<FP8, uint32_t, uint64_t>;
    QP q2[G][DP2];
    const float qscale = a.scale * kLog2e;
    const T* qp = static_cast<const T*>(a.q) + ((size_t)b * a.n_qo_heads + g * G) * D;
    // FP8: each head's q is scaled by a power of two 2^sh that puts its largest magnitude
    // in [2^14, 2^15), inside the f16 range, before the conversion to f16; a bf16 value in
    // f16's normal range converts exactly, and the power of two is exact, so the products
    // see q unchanged up to the values more than 2^24 below the head's largest. 2^-sh then
    // multiplies the dot product. (Without it a |q| above 65504 would become infinite.)
    float q_unscale[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) q_unscale[gi] = 1.0f;
    if constexpr (FP8) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        float mx = 0.0f;
#pragma unroll
        for (int c = 0; c < C::NV; ++c)
#pragma unroll
          for (int e = 0; e < C::VEC; ++e)
            mx = fmaxf(mx, fabsf(to_f32<T>(qp[gi * D + c * C::LPT * C::VEC + j * C::VEC + e])));
#pragma unroll
        for (int off = 1; off < C::LPT; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        // exponent of mx (0 for zero and subnormals), then sh = 14 - exponent, kept inside
        // the normal range of a float scale factor
        const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
        int sh = mx > 0.0f ? 14 - ex : 0;
        sh = sh > 126 ? 126 : (sh < -126 ? -126 : sh);
        const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
        q_unscale[gi] = __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
        for (int c = 0; c < C::NV; ++c)
#pragma unroll
          for (int e = 0; e < C::VEC; e += 2) {
            const T* src = qp + gi * D + c * C::LPT * C::VEC + j * C::VEC + e;
            const __half2 h = __floats2half2_rn(to_f32<T>(src[0]) * up, to_f32<T>(src[1]) * up);
            q2[gi][(c * C::VEC + e) / 2] = *reinterpret_cast<const uint32_t*>(&h);
          }
      }
    } else {
#pragma unroll
      for (int gi = 0; gi < G; ++gi)
#pragma unroll
        for (int c = 0; c < C::NV; ++c)
#pragma unroll
          for (int e = 0; e < C::VEC; e += 2) {
            const T* src = qp + gi * D + c * C::LPT * C::VEC + j * C::VEC + e;
            q2[gi][(c * C::VEC + e) / 2] = pk2(to_f32<T>(src[0]) * qscale, to_f32<T>(src[1]) * qscale);
          }
    }

    const float beta2 = kUnifiedBeta * kLog2e;
    bool first_chunk = true;
    // a head's WPH warps take its pages in turn; every stage is read by one warp per head
    for (int i = warp % C::WPH; i < n_pages; i += C::WPH) {
      const int s = i % C::NSTAGE;
      if (!mbar_wait(bar_full + 8 * s, (i / C::NSTAGE) & 1, a.wait_limit_ns)) {
        if (lane == 0) {
          flags->abort_ = 1;
          set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
        }
        break;
      }
      const KV* kt = reinterpret_cast<const KV*>(smem + s * C::STAGE + hh * C::TILE);
      const KV* vt = reinterpret_cast<const KV*>(smem + (C::NSTAGE + s) * C::STAGE + hh * C::TILE);
      // FP8: this stage's tile scales for the warp's head (1 otherwise; used only for FP8)
      float ks = 1.0f, vs = 1.0f;
      if constexpr (FP8) {
        const float* scl = reinterpret_cast<const float*>(smem + C::SCALE_OFF) + 2 * (C::HPC * s + hh);
        ks = scl[0];
        vs = scl[1];
      }
      const int valid = min(P, kv_len - (first + i) * P);
#pragma unroll
      for (int ch = 0; ch < C::NCHUNK; ++ch) {
        float sc[C::NIT][G];
#pragma unroll
        for (int it = 0; it < C::NIT; ++it) {
          const int t = (ch * C::NIT + it) * C::TPI + tg;
          QP k2[DP2];
#pragma unroll
          for (int c = 0; c < C::NV; ++c) {
            if constexpr (FP8)
              load_row_h2<C::VEC>(kt + t * D + c * C::LPT * C::VEC + j * C::VEC, k2 + c * C::VEC / 2);
            else
              load_row_pairs<KV, C::VEC>(kt + t * D + c * C::LPT * C::VEC + j * C::VEC, k2 + c * C::VEC / 2);
          }
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
            if constexpr (FP8) {
              float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
              for (int e = 0; e < DP2; ++e) fma_h2_f32(q2[gi][e], k2[e], d0, d1);
              sc[it][gi] = ((d0 + d1) * (qscale * ks)) * q_unscale[gi];
            } else {
              uint64_t d2 = 0ull;
#pragma unroll
              for (int e = 0; e < DP2; ++e) d2 = ffma2(q2[gi][e], k2[e], d2);
              const float2 d = upk2(d2);
              sc[it][gi] = d.x + d.y;
            }
          }
        }
        if constexpr (C::SCATTER) {
          // ---- one head per lane: reduce-scatter the dot products, softmax on the lane's
          // own head, then every head's weight for PV from the lanes that own it
          constexpr int LPH = C::LPT / G;  // lanes per head within a token row
          float so[C::NIT];
#pragma unroll
          for (int it = 0; it < C::NIT; ++it) {
            so[it] = reduce_scatter_heads<G, C::LPT>(sc[it], j);
            const int t = (ch * C::NIT + it) * C::TPI + tg;
            if (t >= valid) so[it] = -INFINITY;
          }
          // this chunk's max of head gi, on every lane (lane gi * LPH owns head gi)
          auto chunk_max = [&](float (&mx)[G]) {
            float mo = so[0];
#pragma unroll
            for (int it = 1; it < C::NIT; ++it) mo = fmaxf(mo, so[it]);
#pragma unroll
            for (int off = C::LPT; off < 32; off <<= 1) mo = fmaxf(mo, __shfl_xor_sync(0xffffffffu, mo, off));
#pragma unroll
            for (int gi = 0; gi < G; ++gi) mx[gi] = __shfl_sync(0xffffffffu, mo, gi * LPH);
          };
          auto rescale = [&](int gi, float alpha) {
            const uint64_t al2 = pk2(alpha, alpha);
            if (h_own == gi) lsum_own *= alpha;
#pragma unroll
            for (int e = 0; e < DP2; ++e) acc2[gi][e] = ffma2(acc2[gi][e], al2, 0ull);
          };
          if constexpr (!UNIFIED) {
            float mx[G];
            chunk_max(mx);
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              if (mx[gi] > ref[gi]) {  // warp-uniform
                rescale(gi, ex2(ref[gi] - mx[gi]));
                ref[gi] = mx[gi];
              }
            }
          } else {
            const float ref_o = pick<G>(ref, h_own);
            bool viol = false, all_low = true;
#pragma unroll
            for (int it = 0; it < C::NIT; ++it) {
              viol |= so[it] > ref_o + beta2;
              all_low &= so[it] < ref_o - beta2;
            }
            if (first_chunk) {
              // a head underflows when every lane that owns it saw only low logits
              const unsigned low = __ballot_sync(0xffffffffu, all_low);
#pragma unroll
              for (int gi = 0; gi < G; ++gi) {
                unsigned hm = 0;
#pragma unroll
                for (int r = 0; r < 32 / C::LPT; ++r) hm |= ((1u << LPH) - 1u) << (r * C::LPT + gi * LPH);
                viol |= (low & hm) == hm;
              }
            }
            if (__any_sync(0xffffffffu, viol)) {
              float mx[G];
              chunk_max(mx);
#pragma unroll
              for (int gi = 0; gi < G; ++gi) {
                const bool hi = mx[gi] > ref[gi] + beta2;
                const bool lo = first_chunk && mx[gi] < ref[gi] - beta2;
                if (hi) rescale(gi, ex2(ref[gi] - mx[gi]));
                if (hi || lo) {
                  ref[gi] = mx[gi];
                  ++fallbacks;
                }
              }
            }
            first_chunk = false;
          }
          const float ref_o = pick<G>(ref, h_own);
#pragma unroll
          for (int it = 0; it < C::NIT; ++it) {
            so[it] = ex2(so[it] - ref_o);
            lsum_own += so[it];
          }
#pragma unroll
          for (int it = 0; it < C::NIT; ++it) {
            const int t = (ch * C::NIT + it) * C::TPI + tg;
            float pw[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) pw[gi] = __shfl_sync(0xffffffffu, so[it], tg * C::LPT + gi * LPH);
            QP v2[DP2];
#pragma unroll
            for (int c = 0; c < C::NV; ++c) {
              if constexpr (FP8)
                load_row_h2<C::VEC>(vt + t * D + c * C::LPT * C::VEC + j * C::VEC, v2 + c * C::VEC / 2);
              else
                load_row_pairs<KV, C::VEC>(vt + t * D + c * C::LPT * C::VEC + j * C::VEC, v2 + c * C::VEC / 2);
            }
            if (t < valid) {
#pragma unroll
              for (int gi = 0; gi < G; ++gi) {
                if constexpr (FP8) {
                  const unsigned short ph = f16_bits(pw[gi] * vs);
#pragma unroll
                  for (int e = 0; e < DP2; ++e) acc2[gi][e] = fma_h2s_f32x2(v2[e], ph, acc2[gi][e]);
                } else {
                  const uint64_t p2 = pk2(pw[gi], pw[gi]);
#pragma unroll
                  for (int e = 0; e < DP2; ++e) acc2[gi][e] = ffma2(p2, v2[e], acc2[gi][e]);
                }
              }
            }
          }
        } else {
#pragma unroll
          for (int off = 1; off < C::LPT; off <<= 1)
#pragma unroll
            for (int it = 0; it < C::NIT; ++it)
#pragma unroll
              for (int gi = 0; gi < G; ++gi) sc[it][gi] += __shfl_xor_sync(0xffffffffu, sc[it][gi], off);
#pragma unroll
          for (int it = 0; it < C::NIT; ++it) {
            const int t = (ch * C::NIT + it) * C::TPI + tg;
            if (t >= valid) {
#pragma unroll
              for (int gi = 0; gi < G; ++gi) sc[it][gi] = -INFINITY;
            }
          }

          if constexpr (!UNIFIED) {
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              float mx = sc[0][gi];
#pragma unroll
              for (int it = 1; it < C::NIT; ++it) mx = fmaxf(mx, sc[it][gi]);
#pragma unroll
              for (int off = C::LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
              if (mx > ref[gi]) {  // warp-uniform: every lane holds the same mx and ref
                const float alpha = ex2(ref[gi] - mx);
                const uint64_t al2 = pk2(alpha, alpha);
                ref[gi] = mx;
                lsum[gi] *= alpha;
#pragma unroll
                for (int e = 0; e < DP2; ++e) acc2[gi][e] = ffma2(acc2[gi][e], al2, 0ull);
              }
            }
          } else {
            bool viol = false;
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              bool all_low = true;
#pragma unroll
              for (int it = 0; it < C::NIT; ++it) {
                viol |= sc[it][gi] > ref[gi] + beta2;
                all_low &= sc[it][gi] < ref[gi] - beta2;
              }
              if (first_chunk) viol |= __all_sync(0xffffffffu, all_low);
            }
            if (__any_sync(0xffffffffu, viol)) {
              // Fallback: move each head's reference to this chunk's max where needed.
#pragma unroll
              for (int gi = 0; gi < G; ++gi) {
                float mx = sc[0][gi];
#pragma unroll
                for (int it = 1; it < C::NIT; ++it) mx = fmaxf(mx, sc[it][gi]);
#pragma unroll
                for (int off = C::LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const bool hi = mx > ref[gi] + beta2;
                const bool lo = first_chunk && mx < ref[gi] - beta2;
                if (hi) {
                  // Raise the reference and shrink what was accumulated against the old one.
                  const float alpha = ex2(ref[gi] - mx);
                  const uint64_t al2 = pk2(alpha, alpha);
                  lsum[gi] *= alpha;
#pragma unroll
                  for (int e = 0; e < DP2; ++e) acc2[gi][e] = ffma2(acc2[gi][e], al2, 0ull);
                }
                if (hi || lo) {
                  // A lowered reference (first chunk only) has nothing accumulated to rescale;
                  // ex2(old - new) would overflow there.
                  ref[gi] = mx;
                  ++fallbacks;
                }
              }
            }
            first_chunk = false;
          }

#pragma unroll
          for (int it = 0; it < C::NIT; ++it)
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              sc[it][gi] = ex2(sc[it][gi] - ref[gi]);
              lsum[gi] += sc[it][gi];
            }
#pragma unroll
          for (int it = 0; it < C::NIT; ++it) {
            const int t = (ch * C::NIT + it) * C::TPI + tg;
            QP v2[DP2];
#pragma unroll
            for (int c = 0; c < C::NV; ++c) {
              if constexpr (FP8)
                load_row_h2<C::VEC>(vt + t * D + c * C::LPT * C::VEC + j * C::VEC, v2 + c * C::VEC / 2);
              else
                load_row_pairs<KV, C::VEC>(vt + t * D + c * C::LPT * C::VEC + j * C::VEC, v2 + c * C::VEC / 2);
            }
            if (t < valid) {
#pragma unroll
              for (int gi = 0; gi < G; ++gi) {
                if constexpr (FP8) {
                  const unsigned short ph = f16_bits(sc[it][gi] * vs);
#pragma unroll
                  for (int e = 0; e < DP2; ++e) acc2[gi][e] = fma_h2s_f32x2(v2[e], ph, acc2[gi][e]);
                } else {
                  const uint64_t p2 = pk2(sc[it][gi], sc[it][gi]);
#pragma unroll
                  for (int e = 0; e < DP2; ++e) acc2[gi][e] = ffma2(p2, v2[e], acc2[gi][e]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }

    if constexpr (C::SCATTER) {
#pragma unroll
      for (int off = C::LPT; off < 32; off <<= 1) lsum_own += __shfl_xor_sync(0xffffffffu, lsum_own, off);
#pragma unroll
      for (int gi = 0; gi < G; ++gi) lsum[gi] = __shfl_sync(0xffffffffu, lsum_own, gi * (C::LPT / G));
    }
    // Sum the per-row partials over the token rows of the warp (lanes with equal j).
#pragma unroll
    for (int off = C::LPT; off < 32; off <<= 1)
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        if constexpr (!C::SCATTER) lsum[gi] += __shfl_xor_sync(0xffffffffu, lsum[gi], off);
#pragma unroll
        for (int e = 0; e < DP2; ++e) {
          float2 v = upk2(acc2[gi][e]);
          v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
          v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
          acc2[gi][e] = pk2(v.x, v.y);
        }
      }
  }

  __syncthreads();
  if (flags->abort_) {
    // Wait (bounded) for every copy that was issued, then mark the rows as failed.
    if (threadIdx.x == 0) {
      const int issued = flags->issued;
      for (int s = 0; s < C::NSTAGE && s < issued; ++s) {
        const int last_use = (issued - 1 - s) / C::NSTAGE;
        mbar_wait(bar_full + 8 * s, last_use & 1, a.wait_limit_ns);
      }
    }
    __syncthreads();
    if (final_write) {
      for (int k = 0; k < C::HPC; ++k) write_group_const<T, D, G>(a, b, g0 + k, NAN, NAN);
    } else {
      for (int idx = threadIdx.x; idx < C::HPC * G * D; idx += blockDim.x) {
        const size_t row = (size_t)b * a.n_qo_heads + g0 * G + idx / D;
        a.part_o[(row * a.num_splits + split) * D + idx % D] = NAN;
        if (idx % D == 0) a.part_lse[row * a.num_splits + split] = NAN;
      }
    }
    return;
  }

  // Every issued copy has landed and been consumed: the ring is free for the combine.
  float* cref = reinterpret_cast<float*>(smem);
  float* cl = cref + C::NW * G;
  float* cacc = cl + C::NW * G;
  if (warp < C::NW) {
    if (lane == 0) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        // A warp that accumulated nothing must not set the common reference:
        // in the unified variant its reference is still phi, which may sit far
        // above every real logit.
        cref[warp * G + gi] = lsum[gi] > 0.0f ? ref[gi] : -INFINITY;
        cl[warp * G + gi] = lsum[gi];
      }
      if constexpr (UNIFIED) {
        if (fallbacks) atomicAdd(&flags->fallbacks, fallbacks);
      }
    }
    if (tg == 0) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi)
#pragma unroll
        for (int c = 0; c < C::NV; ++c)
#pragma unroll
          for (int e = 0; e < C::VEC; e += 2) {
            const float2 v = upk2(acc2[gi][(c * C::VEC + e) / 2]);
            cacc[(warp * G + gi) * D + c * C::LPT * C::VEC + j * C::VEC + e] = v.x;
            cacc[(warp * G + gi) * D + c * C::LPT * C::VEC + j * C::VEC + e + 1] = v.y;
          }
    }
  }
  __syncthreads();

  const bool poisoned = flags->bad_page != 0;
  if constexpr (UNIFIED) {
    if (threadIdx.x == 0 && flags->fallbacks && a.fallback_count)
      atomicAdd(a.fallback_count, flags->fallbacks);
  }
  for (int idx = threadIdx.x; idx < C::HPC * G * D; idx += blockDim.x) {
    const int hk = idx / (G * D);  // head within the CTA; its warps are hk*WPH ..
    const int gi = (idx / D) % G;
    const int d = idx % D;
    const int w0 = hk * C::WPH;
    float M = -INFINITY;
#pragma unroll
    for (int w = w0; w < w0 + C::WPH; ++w) M = fmaxf(M, cref[w * G + gi]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = w0; w < w0 + C::WPH; ++w) {
      const float f = ex2(cref[w * G + gi] - M);  // 0 for a warp that saw no page
      L = fmaf(f, cl[w * G + gi], L);
      O = fmaf(f, cacc[(w * G + gi) * D + d], O);
    }
    O = O / L;
    float lse = (M + log2f(L)) * kLn2;
    if (poisoned) {
      O = NAN;
      lse = NAN;
    }
    const int h = (g0 + hk) * G + gi;
    const size_t row = (size_t)b * a.n_qo_heads + h;
    if (final_write) {
      static_cast<T*>(a.out)[row * D + d] = from_f32<T>(O);
      if (a.lse && d == 0) a.lse[row] = lse;
    } else {
      a.part_o[(row * a.num_splits + split) * D + d] = O;
      if (d == 0) a.part_lse[row * a.num_splits + split] = lse;
    }
  }
}

template <typename T, int D, int P, int G, bool UNIFIED, bool FP8 = false>
int launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
  using C = DecodeCfg<T, D, P, G, UNIFIED, FP8>;
  auto kern = decode_paged_kernel<T, D, P, G, UNIFIED, FP8>;
  static FuncConfigured configured;
  if (!configured.ensure(reinterpret_cast<const void*>(kern), C::SMEM)) return PKV_ERR_LAUNCH;
  dim3 grid(a.num_splits, a.n_kv_heads / C::HPC, a.batch);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(a);
  return check_launch(cudaGetLastError());
}

template <typename T, int D, int G, bool FP8 = false>
constexpr int ctas_per_sm_t() {
  using C = DecodeCfg<T, D, 16, G, false, FP8>;
  constexpr int by_smem = (227 * 1024) / C::SMEM;
  return by_smem < C::MIN_BLOCKS ? by_smem : C::MIN_BLOCKS;
}

template <bool UNIFIED>
int dispatch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const int G = a.n_qo_heads / a.n_kv_heads;
#define PKV_DEC_CASE(TT, DD, GG)                                   \
  if (a.head_dim == DD && G == GG)                                 \
    return launch_decode_t<TT, DD, 16, GG, UNIFIED>(a, stream);
#define PKV_DEC_DT(TT)                                             \
  PKV_DEC_CASE(TT, 64, 1) PKV_DEC_CASE(TT, 64, 2) PKV_DEC_CASE(TT, 64, 4) PKV_DEC_CASE(TT, 64, 8) \
  PKV_DEC_CASE(TT, 128, 1) PKV_DEC_CASE(TT, 128, 2)
  if (a.page_size != 16) return PKV_ERR_UNSUPPORTED;
  // bf16 at head_dim 128 with 4 or 8 query heads per KV head runs on the tensor cores
  // (decode_tc.cu) and never reaches this dispatch
  if (a.dtype == PKV_F32) {
    PKV_DEC_DT(float)
    PKV_DEC_CASE(float, 128, 4) PKV_DEC_CASE(float, 128, 8)
  } else if (a.dtype == PKV_BF16) {
    PKV_DEC_DT(__nv_bfloat16)
  }
#undef PKV_DEC_DT
#undef PKV_DEC_CASE
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
