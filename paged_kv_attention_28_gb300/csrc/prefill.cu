// Causal prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Tiled FlashAttention ("快速注意力内核与算子融合", Q&A on FlashAttention): a CTA
// owns two adjacent 128-row query tiles, A and B, of one (batch, head). It
// walks the 128-key K/V tiles up to B's diagonal. For each tile it computes
// S = Q K^T into tensor memory, updates the running row max and sum, writes
// P = exp(S - m) back into tensor memory as bf16, and accumulates O += P V in
// tensor memory. The T x T score matrix never leaves the chip. The causal mask
// is applied by predication on the two diagonal tiles only.
//
// A and B share every K/V tile that TMA brings in. Their softmax work
// alternates with the tensor core: while one warpgroup turns S_A into P_A, the
// tensor core runs B's products, and the other way round.
//
// Warp roles (320 threads):
//   warp 0     TMA producer (Q_A and Q_B once, K/V tiles into a 2-stage ring); owns TMEM
//   warp 1     MMA issuer (one thread)
//   warps 2-5  softmax of tile A, one thread per row (warp w reads TMEM lanes 32*(w%4)..)
//   warps 6-9  softmax of tile B
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// P overwrites the first 64 columns of its own S buffer (packed bf16 pairs).
// PV reads A = P from TMEM and B = V (MN-major) from shared memory.
//
// Lazy rescaling: a row keeps its reference max until a tile's max exceeds it
// by more than 8 (in log2 units). Unnormalised weights then stay <= 2^8, and O
// is rescaled in TMEM only on those rare tiles. The final O / l is exact either way.
//
// The same kernel, instantiated with CAUSAL = false, is the shared-prefix
// ("cascade") kernel. There a 128-row query tile is 128/G requests x the G query
// heads of one KV head, and K/V tiles are gathered 16 rows (one page) at a time
// through the prefix block table. The prefix is cut into chunks of key tiles,
// one chunk per CTA, and each CTA writes fp32 partial (O, LSE) states that a
// later merge combines with the per-request suffix.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
constexpr int HD = 128;        // head dim
constexpr int SUB = 16384;     // one 128-row x 64-column bf16 sub-tile (128-byte swizzle)
constexpr int TILE = 2 * SUB;  // 128 x 128 bf16
constexpr int NST = 2;         // K/V ring stages
constexpr int SM_Q = 0;                      // Q_A, Q_B
constexpr int SM_K = SM_Q + 2 * TILE;
constexpr int SM_V = SM_K + NST * TILE;
constexpr int SM_BAR = SM_V + NST * TILE;
// barriers: q_full, kv_full[2], kv_empty[2], s_full[2], p_full[2], o_done[2], drain
constexpr int BAR_Q = 0, BAR_KVF = 1, BAR_KVE = 3, BAR_SF = 5, BAR_PF = 7, BAR_OD = 9,
              BAR_DRAIN = 11, NBAR = 12;
constexpr int SM_MISC = SM_BAR + NBAR * 8;
constexpr int SMEM_BYTES = SM_MISC + 64 + 1024;  // + slack to align the base to 1024
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr int COL_S = 0, COL_O = 256;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;  // log2 units

struct Misc {
  uint32_t tmem_base;
  int abort_;
  int bad_page;
};

// Everything either instantiation needs.
struct TileArgs {
  void* out;          // causal: bf16 [B, T, Hq, D]
  float* lse;         // causal: fp32 [B, Hq, T] (nullable)
  int32_t* err_flag;
  float scale;
  int batch, seq_len, n_qo_heads, n_kv_heads;
  // shared prefix
  const int32_t* prefix_table;
  int prefix_len, n_prefix_pages, n_requests, num_pages;
  int tiles_per_chunk, n_chunks, n_row_pairs;
  float* part_o;      // fp32 [n_chunks][n_requests][Hq][D]
  float* part_lse;    // fp32 [n_chunks][n_requests][Hq]
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}

// A wait taken by every lane of a warp; the result is the same on all lanes, so
// the .sync.aligned tcgen05 instructions that follow never diverge.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void fail(Misc* misc, int32_t* err) {
  misc->abort_ = 1;
  set_err(err, PKV_DEVERR_TIMEOUT);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Where a query tile's rows go and which keys its last tile may use.
struct TileJob {
  int n_tiles;     // key tiles this query tile walks
  int last_valid;  // keys usable in its last key tile (prefix); unused when causal
  // causal: output rows t = q0 + r of (b, h)
  int q0, b, h;
  // prefix: row r of the tile is request r0 + r / G, query head g*G + r % G, chunk c
  int r0, g, c;
};

// The softmax warpgroup of one query tile: S -> P for every key tile, then the epilogue.
template <bool CAUSAL>
__device__ __forceinline__ void softmax_tile(const TileArgs& a, Misc* misc, uint32_t bar_sf,
                                             uint32_t bar_pf, uint32_t bar_od, uint32_t col_s,
                                             uint32_t col_o, const TileJob& job, int warp, int lane) {
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // row in the tile = TMEM lane
  const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
  const uint32_t tS = misc->tmem_base + lane_addr + col_s;
  const uint32_t tO = misc->tmem_base + lane_addr + col_o;
  const float c = a.scale * kLog2eF;  // logits in log2 units: s * c
  float ms = -INFINITY;               // reference max, log2 units
  float l = 0.0f;
  bool ok = true;
  const int n_tiles = job.n_tiles;
  for (int jj = 0; jj < n_tiles; ++jj) {
    if (!warp_wait(bar_sf, jj & 1)) { ok = false; break; }
    tc_fence_after();
    uint32_t sr[128];
    tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(sr + 0));
    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(sr + 64));
    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(sr + 96));
    tmem_ld_wait();
    float* x = reinterpret_cast<float*>(sr);
    if (jj == n_tiles - 1) {
      // causal: key column i is visible to row r iff i <= r (diagonal tile);
      // prefix: only the first last_valid keys of the last tile exist
      const int limit = CAUSAL ? r + 1 : job.last_valid;
#pragma unroll
      for (int i = 0; i < 128; ++i) x[i] = (i >= limit) ? -INFINITY : x[i];
    }
    float mx = fmaxf(x[0], x[1]);
#pragma unroll
    for (int i = 2; i < 128; i += 2) mx = max3(mx, x[i], x[i + 1]);
    const float mt = mx * c;
    const bool need = mt > ms + kRescaleSlack;  // always on the first tile (ms = -inf)
    const float m_new = need ? mt : ms;
    const float alpha = need ? ex2(ms - m_new) : 1.0f;
    const uint64_t cc = f2(c, c);
    const uint64_t mm = f2(-m_new, -m_new);
    uint64_t acc = f2(0.0f, 0.0f);
    uint32_t pk[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      float y0, y1;
      unf2(fma2(f2(x[2 * i], x[2 * i + 1]), cc, mm), y0, y1);
      const float p0 = ex2(y0), p1 = ex2(y1);
      acc = add2(acc, f2(p0, p1));
      pk[i] = pack_bf16x2(p0, p1);
    }
    float s0, s1;
    unf2(acc, s0, s1);
    l = l * alpha + (s0 + s1);
    // S_j's completion implies PV_{j-1} has completed (the commit for S_j was
    // issued after it), so O is stable here and P's columns are free.
    if (jj > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t o[32];
        tmem_ld32(tO + q * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tO + q * 32, o);
      }
    }
    ms = m_new;
    tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(pk + 0));
    tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar_pf);
  }
  // ------------------------------------------------------------------ epilogue
  ok = __all_sync(0xffffffffu, ok);
  if (ok && !warp_wait(bar_od, (n_tiles - 1) & 1)) ok = false;
  tc_fence_after();
  if (!ok && lane == 0) fail(misc, a.err_flag);
  if (*reinterpret_cast<volatile int*>(&misc->bad_page)) ok = false;
  const float inv = ok ? 1.0f / l : NAN;
  const float lse_row = ok ? (ms + log2f(l)) * kLn2F : NAN;
  const int H = a.n_qo_heads;
  if constexpr (CAUSAL) {
    const int t = job.q0 + r;
    const bool store = t < a.seq_len;  // rows past a ragged end are computed but not stored
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(a.out) + (((size_t)job.b * a.seq_len + t) * H + job.h) * HD;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o[32];
      tmem_ld32(tO + q * 32, o);  // all lanes, uniformly
      tmem_ld_wait();
      uint4 w[4];
      uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        wp[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = w[i];
      }
    }
    if (store && a.lse) a.lse[((size_t)job.b * H + job.h) * a.seq_len + t] = lse_row;
  } else {
    const int G = a.n_qo_heads / a.n_kv_heads;
    const int req = job.r0 + r / G;
    const int h = job.g * G + r % G;
    const bool store = req < a.n_requests;
    const size_t row = ((size_t)job.c * a.n_requests + req) * H + h;
    float* orow = a.part_o + row * HD;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o[32];
      tmem_ld32(tO + q * 32, o);
      tmem_ld_wait();
      if (store) {
        float4* dst = reinterpret_cast<float4*>(orow + q * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                               __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
      }
    }
    if (store) a.part_lse[row] = lse_row;
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
attn_tile_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const TileArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  Misc* misc = reinterpret_cast<Misc*>(smem + SM_MISC);
  auto bar = [&](int i) { return sb + SM_BAR + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.n_qo_heads;
  const int G = a.n_qo_heads / a.n_kv_heads;
  const int id = blockIdx.x;

  // ---------------------------------------------------------------- what this CTA does
  TileJob jobA{}, jobB{};
  bool has_b;
  int n_kv;      // key tiles the CTA walks
  int lastA;     // A's last key tile
  int kv_first;  // prefix: first key tile of the chunk
  int hk, qrow;  // KV head; causal: first query row of A
  if constexpr (CAUSAL) {
    const int n_qt = (a.seq_len + BM - 1) / BM;
    const int n_pairs = (n_qt + 1) / 2;
    // Longest-first order: the pairs nearest the end of the sequence have the most key tiles.
    const int pr = n_pairs - 1 - id / (H * a.batch);
    const int rem = id % (H * a.batch);
    const int h = rem % H;
    const int b = rem / H;
    hk = h / G;
    const int qtA = 2 * pr;
    has_b = (qtA + 1) < n_qt;
    lastA = qtA;
    n_kv = has_b ? qtA + 2 : qtA + 1;
    kv_first = 0;
    qrow = qtA * BM;
    jobA = TileJob{qtA + 1, BN, qtA * BM, b, h, 0, 0, 0};
    jobB = TileJob{qtA + 2, BN, (qtA + 1) * BM, b, h, 0, 0, 0};
  } else {
    const int c = id % a.n_chunks;
    const int rest = id / a.n_chunks;
    hk = rest % a.n_kv_heads;
    const int pr = rest / a.n_kv_heads;
    const int n_tiles = (a.n_prefix_pages + 7) / 8;
    kv_first = c * a.tiles_per_chunk;
    n_kv = min(a.tiles_per_chunk, n_tiles - kv_first);
    lastA = n_kv - 1;
    has_b = (pr * 2 * BM + BM) < a.n_requests * G;
    qrow = pr * 2 * BM;  // row of the (request, head-in-group) list
    const int last_valid = a.prefix_len - (kv_first + n_kv - 1) * BN;
    jobA = TileJob{n_kv, last_valid, 0, 0, 0, qrow / G, hk, c};
    jobB = TileJob{n_kv, last_valid, 0, 0, 0, (qrow + BM) / G, hk, c};
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == BAR_PF || i == BAR_PF + 1) ? 128 : 1);
    misc->abort_ = 0;
    misc->bad_page = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      mbar_arrive_expect_tx(bar(BAR_Q), 2 * TILE);
      for (int t = 0; t < 2; ++t) {
        for (int half = 0; half < 2; ++half) {
          const uint32_t dst = sb + SM_Q + t * TILE + half * SUB;
          if constexpr (CAUSAL)
            tma_load_4d(dst, &mq, half * 64, jobA.h, qrow + t * BM, jobA.b, bar(BAR_Q));
          else
            tma_load_3d(dst, &mq, half * 64, hk * G, (qrow + t * BM) / G, bar(BAR_Q));
        }
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NST, u = j / NST;
        if (u > 0 && !mbar_wait(bar(BAR_KVE + s), (u - 1) & 1)) {
          fail(misc, a.err_flag);
          break;
        }
        if (misc->abort_) break;
        mbar_arrive_expect_tx(bar(BAR_KVF + s), 2 * TILE);
        const uint32_t dk = sb + SM_K + s * TILE, dv = sb + SM_V + s * TILE;
        if constexpr (CAUSAL) {
          const int k0 = j * BN;
          tma_load_4d(dk, &mk, 0, hk, k0, jobA.b, bar(BAR_KVF + s));
          tma_load_4d(dk + SUB, &mk, 64, hk, k0, jobA.b, bar(BAR_KVF + s));
          tma_load_4d(dv, &mv, 0, hk, k0, jobA.b, bar(BAR_KVF + s));
          tma_load_4d(dv + SUB, &mv, 64, hk, k0, jobA.b, bar(BAR_KVF + s));
        } else {
          // Eight pages of 16 keys make one 128-key tile; each page is a 16-row box.
          // Slots past the prefix reload its first page (finite data; masked out).
          for (int pp = 0; pp < 8; ++pp) {
            const int page_idx = (kv_first + j) * 8 + pp;
            int phys = __ldg(a.prefix_table + (page_idx < a.n_prefix_pages ? page_idx : 0));
            if (phys < 0 || phys >= a.num_pages) {
              misc->bad_page = 1;
              set_err(a.err_flag, PKV_DEVERR_BAD_PAGE);
              phys = 0;
            }
            const int row = (phys * a.n_kv_heads + hk) * 16;
            tma_load_2d(dk + pp * 2048, &mk, 0, row, bar(BAR_KVF + s));
            tma_load_2d(dk + SUB + pp * 2048, &mk, 64, row, bar(BAR_KVF + s));
            tma_load_2d(dv + pp * 2048, &mv, 0, row, bar(BAR_KVF + s));
            tma_load_2d(dv + SUB + pp * 2048, &mv, 64, row, bar(BAR_KVF + s));
          }
        }
        issued = j + 1;
      }
      // Every issued copy must land before the CTA's shared memory is released
      // (immediate on the normal path, where the MMA warp already waited for them).
      if (!mbar_wait(bar(BAR_Q), 0)) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
      for (int s = 0; s < NST && s < issued; ++s)
        if (!mbar_wait(bar(BAR_KVF + s), ((issued - 1 - s) / NST) & 1))
          set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
      const uint32_t idPV = idesc_bf16_f32(BM, HD, false, true);
      auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T
        const uint32_t kb = sb + SM_K + (j % NST) * TILE;
        const uint32_t qb = sb + SM_Q + t * TILE;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k / 4) * SUB + (k % 4) * 32;
          mma_bf16_ss(tmem + COL_S + t * BN, smem_desc(qb + off, 16, 1024, kSwizzle128B),
                      smem_desc(kb + off, 16, 1024, kSwizzle128B), idS, k > 0);
        }
        mma_commit(bar(BAR_SF + t));
      };
      auto issue_pv = [&](int t, int j) {  // O_t += P_t V_j
        const uint32_t vb = sb + SM_V + (j % NST) * TILE;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ts(tmem + COL_O + t * HD, tmem + COL_S + t * BN + k * 8,
                      smem_desc(vb + k * 2048, 16384, 1024, kSwizzle128B), idPV,
                      (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(BAR_OD + t));
      };
      bool ok = mbar_wait(bar(BAR_Q), 0) && mbar_wait(bar(BAR_KVF + 0), 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (has_b) issue_s(1, 0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j <= lastA) {
          if (!mbar_wait(bar(BAR_PF + 0), j & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, j);
        }
        if (j + 1 < n_kv) {
          if (!mbar_wait(bar(BAR_KVF + (j + 1) % NST), ((j + 1) / NST) & 1)) { ok = false; break; }
          tc_fence_after();
          if (j + 1 <= lastA) issue_s(0, j + 1);
        }
        if (has_b) {
          if (!mbar_wait(bar(BAR_PF + 1), j & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, j);
        }
        mma_commit(bar(BAR_KVE + j % NST));  // K_j / V_j are no longer read by any product
        if (has_b && j + 1 < n_kv) issue_s(1, j + 1);
      }
      if (!ok) fail(misc, a.err_flag);
      // Every issued product must finish before TMEM is freed.
      mma_commit(bar(BAR_DRAIN));
      if (!mbar_wait(bar(BAR_DRAIN), 0)) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp < 6) {
    softmax_tile<CAUSAL>(a, misc, bar(BAR_SF + 0), bar(BAR_PF + 0), bar(BAR_OD + 0), COL_S, COL_O,
                         jobA, warp, lane);
  } else if (has_b) {
    softmax_tile<CAUSAL>(a, misc, bar(BAR_SF + 1), bar(BAR_PF + 1), bar(BAR_OD + 1), COL_S + BN,
                         COL_O + HD, jobB, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B, T, H, D] bf16 viewed as a 4-D tensor (D, H, T, B); a box is 64 columns x 128 rows of one head.
bool make_btHd_map(CUtensorMap* m, const void* ptr, int B, int T, int H) {
  cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)H * HD * 2, (cuuint64_t)T * H * HD * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  return encode(m, ptr, 4, dims, strides, box);
}

template <bool CAUSAL>
int launch_tiles(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                 const TileArgs& a, long grid, cudaStream_t stream) {
  if (grid <= 0) return PKV_OK;
  if (grid > 0x7fffffffL) return PKV_ERR_UNSUPPORTED;
  static int configured_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 32 && !(configured_mask & (1 << dev))) {
    if (check_launch(cudaFuncSetAttribute(attn_tile_kernel<CAUSAL>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)) != PKV_OK)
      return PKV_ERR_LAUNCH;
    configured_mask |= (1 << dev);
  }
  attn_tile_kernel<CAUSAL><<<(unsigned)grid, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, a);
  return check_launch(cudaGetLastError());
}

}  // namespace

int launch_prefill(const PrefillArgs& p, cudaStream_t stream) {
  if (p.head_dim != HD) return PKV_ERR_UNSUPPORTED;
  const long n_qt = (p.seq_len + BM - 1) / BM;
  const long grid = (n_qt + 1) / 2 * p.n_qo_heads * p.batch;
  CUtensorMap mq, mk, mv;
  if (!make_btHd_map(&mq, p.q, p.batch, p.seq_len, p.n_qo_heads) ||
      !make_btHd_map(&mk, p.k, p.batch, p.seq_len, p.n_kv_heads) ||
      !make_btHd_map(&mv, p.v, p.batch, p.seq_len, p.n_kv_heads))
    return check_launch(cudaErrorInvalidValue);
  TileArgs a{};
  a.out = p.out;
  a.lse = p.lse;
  a.err_flag = p.err_flag;
  a.scale = p.scale;
  a.batch = p.batch;
  a.seq_len = p.seq_len;
  a.n_qo_heads = p.n_qo_heads;
  a.n_kv_heads = p.n_kv_heads;
  return launch_tiles<true>(mq, mk, mv, a, grid, stream);
}

// Tensor-core prefix attention of the cascade path: fp32 partial states per prefix chunk.
int launch_cascade_prefix(const CascadeArgs& c, cudaStream_t stream) {
  if (c.head_dim != HD || c.page_size != 16) return PKV_ERR_UNSUPPORTED;
  const int G = c.n_qo_heads / c.n_kv_heads;
  if (BM % G) return PKV_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  {
    // q [R, Hq, D] as (D, Hq, R): one box = G heads x 128/G requests = 128 rows of 64 columns
    cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)c.n_qo_heads, (cuuint64_t)c.n_requests};
    cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)c.n_qo_heads * HD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(BM / G)};
    if (!encode(&mq, c.q, 3, dims, strides, box)) return check_launch(cudaErrorInvalidValue);
  }
  {
    // pools [pages, Hkv, 16, D] as rows of D: one box = one (page, head) tile, 16 rows x 64 columns
    const cuuint64_t rows = (cuuint64_t)c.num_pages * c.n_kv_heads * 16;
    cuuint64_t dims[2] = {(cuuint64_t)HD, rows};
    cuuint64_t strides[1] = {(cuuint64_t)HD * 2};
    cuuint32_t box[2] = {64, 16};
    if (!encode(&mk, c.k_pages, 2, dims, strides, box) || !encode(&mv, c.v_pages, 2, dims, strides, box))
      return check_launch(cudaErrorInvalidValue);
  }
  TileArgs a{};
  a.err_flag = c.err_flag;
  a.scale = c.scale;
  a.n_qo_heads = c.n_qo_heads;
  a.n_kv_heads = c.n_kv_heads;
  a.prefix_table = c.prefix_table;
  a.prefix_len = c.prefix_len;
  a.n_prefix_pages = c.prefix_len / 16;
  a.n_requests = c.n_requests;
  a.num_pages = c.num_pages;
  const int n_tiles = (a.n_prefix_pages + 7) / 8;
  a.n_chunks = c.prefix_chunks;
  a.tiles_per_chunk = (n_tiles + a.n_chunks - 1) / a.n_chunks;
  a.n_chunks = (n_tiles + a.tiles_per_chunk - 1) / a.tiles_per_chunk;  // no empty chunk
  a.n_row_pairs = (c.n_requests * G + 2 * BM - 1) / (2 * BM);
  a.part_o = c.pre_o;
  a.part_lse = c.pre_lse;
  if (a.n_chunks != c.prefix_chunks) return PKV_ERR_INVALID_ARG;  // planner guarantees equality
  const long grid = (long)a.n_chunks * c.n_kv_heads * a.n_row_pairs;
  return launch_tiles<false>(mq, mk, mv, a, grid, stream);
}

}  // namespace pkv
