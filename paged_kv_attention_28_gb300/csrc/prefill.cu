// Causal prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Tiled FlashAttention ("快速注意力内核与算子融合", Q&A on FlashAttention): a work
// item is two adjacent 128-row query tiles, A and B, of one (batch, head). A CTA
// walks the item's 128-key K/V tiles up to B's diagonal, each in two steps of 64 keys. For
// each step it computes S = Q K^T into tensor memory, updates the running row max and
// sum, writes P = exp(S - m) back into tensor memory as bf16, and accumulates O += P V
// in tensor memory. The T x T score matrix never leaves the chip. The causal mask is
// applied by predication on the two diagonal tiles only.
//
// The grid has one CTA per item; a running CTA also takes the items of CTAs that have
// not started yet (cluster launch control, below), so one CTA per SM runs to the end.
//
// A and B share every K/V tile that TMA brings in. Each query tile has two S buffers,
// so S for step s + 1 is computed while the softmax turns S_s into P_s: the chain
// S -> softmax -> PV -> S that would otherwise serialise a tile is cut in two, and
// the two tiles' products and softmaxes overlap.
//
// Warp roles (512 threads, four warpgroups):
//   warpgroup 0: warp 0 TMA producer of Q_A, Q_B (per item) and K tiles (2-stage ring;
//                owns TMEM), warp 3 TMA producer of V tiles (3-stage ring), warps 1 and
//                2 MMA issuers of tiles A and B. All four run their loops as whole warps
//                and issue from an elected lane.
//   warpgroup 1: softmax of tile A, one thread per row (warp w reads TMEM lanes 32*(w%4)..)
//   warpgroup 2: softmax of tile B
//   warpgroup 3: epilogue: O / l out of TMEM to global memory, for both tiles
// Registers are rebalanced with setmaxnreg: the softmax warpgroups get 168 per thread,
// the other two 88 (88 + 168 + 168 + 88 = 512 per SM sub-partition, the launch's share).
// TMEM columns: S_A,0 [0,64), S_A,1 [64,128), S_B,0 [128,192), S_B,1 [192,256),
// O_A [256,384), O_B [384,512). P overwrites the first 32 columns of its own S buffer
// (packed bf16 pairs).
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
// one chunk per item, and each item writes fp32 partial (O, LSE) states that a
// later merge combines with the per-request suffix.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "internal.h"
#include "tcgen05.cuh"
#include "work_queue.cuh"

namespace pkv {
namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per K/V tile
constexpr int BS = 64;         // keys per S step (half a K/V tile)
constexpr int HD = 128;        // head dim
constexpr int SUB = 16384;     // one 128-row x 64-column bf16 sub-tile (128-byte swizzle)
constexpr int TILE = 2 * SUB;  // 128 x 128 bf16
constexpr int NSK = 2;         // K ring stages (a K tile is free once both S products read it)
constexpr int NSV = 3;         // V ring stages (a V tile is free once both PV products read it)
constexpr int kReqAhead = 1;   // K tiles of an item still to copy when the next item is requested
constexpr int NQ = 2;          // Q buffers: Q tile n (item k, tile t: n = 2k + t) uses buffer n % NQ
constexpr int NQB = 2 * NQ;    // q_full / q_empty barriers: tile n uses barrier n % NQB
constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + NQ * TILE;
constexpr int SM_V = SM_K + NSK * TILE;
constexpr int SM_BAR = SM_V + NSV * TILE;
// Barriers. q_full / q_empty: Q tile n uses barrier n % NQB, so each barrier serves one MMA
// issuer (tile n % 2) in turn and every wait on it is for the phase after the last one that
// issuer saw. k_full / k_empty, v_full / v_empty: the rings (empty takes one arrival from each
// MMA issuer). s_full[2 tiles][2 buffers], p_full[2][2]; o_done[2] (one phase per PV step);
// drain[2]; o_free[2] (the epilogue read O); st_full[2] (a tile's softmax wrote its rows' 1/l
// for the epilogue warpgroup); inv_empty[2] (the epilogue read them, so the next item's
// softmax may overwrite them); o_item[2] (an item's last PV finished); next_full[NXS] /
// next_empty[NXS]: the ring of work-distribution responses (work_queue.cuh), next_full
// completing when a response lands (16 bytes) and next_empty taking one arrival from every
// warp; v_zeroed (chunk mode): tile B's issuer has zeroed the V rows past the sequence's end
// in the last key tile that both tiles read (one phase per such item).
constexpr int BAR_QF = 0, BAR_QE = BAR_QF + NQB, BAR_KF = BAR_QE + NQB, BAR_KE = BAR_KF + NSK,
              BAR_VF = BAR_KE + NSK, BAR_VE = BAR_VF + NSV, BAR_SF = BAR_VE + NSV, BAR_PF = BAR_SF + 4,
              BAR_OD = BAR_PF + 4, BAR_DRAIN = BAR_OD + 2, BAR_OF = BAR_DRAIN + 2, BAR_ST = BAR_OF + 2,
              BAR_IE = BAR_ST + 2, BAR_OI = BAR_IE + 2, BAR_NF = BAR_OI + 2, BAR_NE = BAR_NF + NXS,
              BAR_VZ = BAR_NE + NXS;
constexpr int NBAR = (BAR_VZ + 2) & ~1;  // even, so that what follows is 16-byte aligned
constexpr int SM_INV = SM_BAR + NBAR * 8;          // float [2 tiles][128 rows]: 1/l per row
constexpr int SM_MISC = SM_INV + 2 * BM * 4;
constexpr int SMEM_BYTES = SM_MISC + 128 + 1024;  // + slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr int THREADS = 512;  // four warpgroups; see the role list at the top
constexpr int TMEM_COLS = 512;
constexpr int COL_S = 0, COL_O = 256;  // tile t: S buffers at t*128 + b*64, O at COL_O + t*128
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;  // log2 units

constexpr int NBAD = 8;  // bad-page marks kept for the last NBAD items of a CTA
struct Misc {
  uint4 next[NXS];  // responses of the work-distribution requests (16-byte aligned)
  uint32_t tmem_base;
  int abort_;
  // bad_item[k % NBAD] holds the id of this CTA's k-th item if one of its table entries
  // was out of range. Ids are unique within a launch, so a mark left by item k - NBAD
  // never matches item k; a producer is never NBAD items ahead of the softmax warps
  // (each item's request for the next one waits for every warp to finish item k - NXS).
  int bad_item[NBAD];
};
static_assert(sizeof(Misc) <= 128 && SM_MISC % 16 == 0, "Misc layout");

// Everything either instantiation needs.
struct TileArgs {
  void* out;          // causal: bf16 [B, T, Hq, D]
  float* lse;         // causal: fp32 [B, Hq, T] (nullable)
  int32_t* err_flag;
  float scale;
  int batch, seq_len, n_qo_heads, n_kv_heads;
  int group_bh, tail_bh;  // causal and chunk item order (grouped_order)
  // shared prefix
  const int32_t* prefix_table;
  int prefix_len, n_prefix_pages, n_requests, num_pages;
  int tiles_per_chunk, n_chunks, n_row_pairs;
  float* part_o;      // fp32 [n_chunks][n_requests][Hq][D]
  float* part_lse;    // fp32 [n_chunks][n_requests][Hq]
  // chunked prefill over the paged cache: C new tokens per sequence after prefix_lens[b]
  const int32_t* block_table;  // int32 [batch][max_blocks]
  const int32_t* prefix_lens;  // int32 [batch]
  int chunk_len, max_blocks;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
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
  int n_tiles;     // key tiles this query tile walks (0: the tile does not exist)
  int last_valid;  // keys usable in its last key tile (prefix); unused when causal
  // causal: output rows t = q0 + r of (b, h)
  int q0, b, h;
  // prefix: row r of the tile is request r0 + r / G, query head g*G + r % G, chunk c
  int r0, g, c;
  // chunk: row r is new token q0 + r / G (position L0 + q0 + r / G) of sequence b, query
  // head g*G + r % G
  int L0;
};

// One work item: two query tiles (A, B) that share their key tiles.
struct Item {
  TileJob A, B;
  int n_kv;      // key tiles the item walks (B's count when B exists)
  int kv_first;  // prefix: first key tile of the chunk
  int hk;        // KV head
  int qrow;      // causal: first query row of A; prefix: first (request, head) row of A
  int b;         // causal: batch
  int id;        // the item's index in the grid
};

// Item order for work made of `units` units (a (b, h) or (b, KV head)) of n_pairs query-tile
// pairs each, pair n_pairs - 1 the longest (CTAs take items in index order): the units but
// the last `tail` go in groups of `group`, each group's pairs longest first, so that the
// pairs reading the same K/V run at about the same time and find it in L2; the last `tail`
// units go longest first over all their pairs, so the grid ends on short items.
__device__ __forceinline__ void grouped_order(int id, int units, int n_pairs, int group, int tail_units,
                                              int& pr, int& unit) {
  const int tail = min(units, tail_units);
  const int head_items = (units - tail) * n_pairs;
  if (id < head_items) {
    const int per_group = group * n_pairs;
    const int gi = id / per_group;
    const int gsz = min(group, (units - tail) - gi * group);
    const int rr = id - gi * per_group;
    pr = n_pairs - 1 - rr / gsz;
    unit = gi * group + rr % gsz;
  } else {
    const int rr = id - head_items;
    pr = n_pairs - 1 - rr / tail;
    unit = (units - tail) + rr % tail;
  }
}

template <bool CAUSAL, bool CHUNK = false>
__device__ __forceinline__ Item make_item(const TileArgs& a, int id) {
  Item it{};
  it.id = id;
  const int H = a.n_qo_heads;
  const int G = a.n_qo_heads / a.n_kv_heads;
  if constexpr (CHUNK) {
    // Items (query-tile pair, KV head, sequence) in grouped_order over the (sequence, KV
    // head) units: every pair of a unit reads the unit's whole prefix, so a unit's pairs run
    // at about the same time and the prefix's K/V comes from L2 after the first.
    // A tile is 128/G new tokens x the G query heads of one KV head.
    const int TPT = BM / G;  // tokens per tile
    const int n_qt = (a.chunk_len + TPT - 1) / TPT;
    const int n_pairs = (n_qt + 1) / 2;
    int pr, rem;
    grouped_order(id, a.batch * a.n_kv_heads, n_pairs, a.group_bh, a.tail_bh, pr, rem);
    const int hk = rem % a.n_kv_heads;
    const int b = rem / a.n_kv_heads;
    int L0 = __ldg(a.prefix_lens + b);
    const int cap = a.max_blocks * 16 - a.chunk_len;
    if (L0 < 0 || L0 > cap) {  // reported; the rows are then computed on a clamped length
      set_err(a.err_flag, PKV_DEVERR_BAD_LEN);
      L0 = L0 < 0 ? 0 : cap;
    }
    const int q0A = 2 * pr * TPT, q0B = q0A + TPT;
    const bool has_b = q0B < a.chunk_len;
    // key tiles up to the last real token of the tile (position L0 + last)
    auto tiles = [&](int q0) { return (L0 + min(q0 + TPT, a.chunk_len) + BN - 1) / BN; };
    it.hk = hk;
    it.b = b;
    it.A = TileJob{tiles(q0A), 0, q0A, b, 0, 0, hk, 0, L0};
    it.B = TileJob{has_b ? tiles(q0B) : 0, 0, q0B, b, 0, 0, hk, 0, L0};
    it.n_kv = has_b ? it.B.n_tiles : it.A.n_tiles;
  } else if constexpr (CAUSAL) {
    const int n_qt = (a.seq_len + BM - 1) / BM;
    const int n_pairs = (n_qt + 1) / 2;
    // Items in grouped_order over the (b, h) units; the pairs nearest the end of the
    // sequence have the most key tiles.
    int pr, rem;
    grouped_order(id, H * a.batch, n_pairs, a.group_bh, a.tail_bh, pr, rem);
    const int h = rem % H;
    const int b = rem / H;
    const int qtA = 2 * pr;
    const bool has_b = (qtA + 1) < n_qt;
    it.hk = h / G;
    it.b = b;
    it.n_kv = has_b ? qtA + 2 : qtA + 1;
    it.qrow = qtA * BM;
    it.A = TileJob{qtA + 1, BN, qtA * BM, b, h, 0, 0, 0, 0};
    it.B = TileJob{has_b ? qtA + 2 : 0, BN, (qtA + 1) * BM, b, h, 0, 0, 0, 0};
  } else {
    const int c = id % a.n_chunks;
    const int rest = id / a.n_chunks;
    const int hk = rest % a.n_kv_heads;
    const int pr = rest / a.n_kv_heads;
    const int n_tiles = (a.n_prefix_pages + 7) / 8;
    it.hk = hk;
    it.kv_first = c * a.tiles_per_chunk;
    it.n_kv = min(a.tiles_per_chunk, n_tiles - it.kv_first);
    const bool has_b = (pr * 2 * BM + BM) < a.n_requests * G;
    it.qrow = pr * 2 * BM;
    const int last_valid = a.prefix_len - (it.kv_first + it.n_kv - 1) * BN;
    it.A = TileJob{it.n_kv, last_valid, 0, 0, 0, it.qrow / G, hk, c, 0};
    it.B = TileJob{has_b ? it.n_kv : 0, last_valid, 0, 0, 0, (it.qrow + BM) / G, hk, c, 0};
  }
  return it;
}

// The softmax warpgroup of one query tile of every item of this CTA: S -> P for each
// 64-key step, then the hand-off to the epilogue. Step g of the tile (counted across
// items) uses S buffer g & 1 and barriers s_full[g & 1], p_full[g & 1].
template <bool CAUSAL, bool CHUNK = false>
__device__ __forceinline__ void softmax_loop(const TileArgs& a, Misc* misc, uint32_t bar_sf0,
                                             uint32_t bar_pf0, uint32_t bar_od, uint32_t bar_st,
                                             uint32_t bar_ie, float* inv_rows,
                                             uint32_t col_s, uint32_t col_o, int tile, int n_items,
                                             const NextRing& ring, int warp, int lane) {
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // row in the tile = TMEM lane
  const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
  const uint32_t tS = misc->tmem_base + lane_addr + col_s;
  const uint32_t tO = misc->tmem_base + lane_addr + col_o;
  const float c = a.scale * kLog2eF;  // logits in log2 units: s * c
  const int H = a.n_qo_heads;
  uint32_t g = 0, st_cnt = 0;  // steps done (across items); items handed off
  bool ok = true;
  uint32_t k = 0;
  for (int id = blockIdx.x; id < n_items; id = next_item(ring, k++, n_items, a.err_flag)) {
    const Item it = make_item<CAUSAL, CHUNK>(a, id);
    const TileJob& job = tile == 0 ? it.A : it.B;
    const int n_steps = 2 * job.n_tiles;
    if (n_steps == 0) continue;
    float ms = -INFINITY;  // reference max, log2 units
    float l = 0.0f;
    for (int s = 0; s < n_steps; ++s, ++g) {
      const uint32_t b = g & 1;
      if (ok && !warp_wait(bar_sf0 + 8 * b, (g >> 1) & 1)) ok = false;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tSb = tS + b * BS;
      uint32_t sr[BS];
      tmem_ld32(tSb + 0, *reinterpret_cast<uint32_t(*)[32]>(sr + 0));
      tmem_ld32(tSb + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_ld_wait();
      float* x = reinterpret_cast<float*>(sr);
      if constexpr (CHUNK) {
        // row r (position L0 + q0 + r/G) sees keys up to its own position; the step holds
        // keys [64 s, 64 s + 64)
        const int first_pos = job.L0 + job.q0;  // the tile's smallest position
        if (s * BS + BS > first_pos + 1) {
          const int G = a.n_qo_heads / a.n_kv_heads;
          const int limit = first_pos + r / G + 1 - s * BS;
#pragma unroll
          for (int i = 0; i < BS; ++i) x[i] = (i >= limit) ? -INFINITY : x[i];
        }
      } else if (s >= n_steps - 2) {
        // causal: key column k of the tile is visible to row r iff k <= r (diagonal
        // tile); prefix: only the first last_valid keys of the last tile exist
        const int limit = (CAUSAL ? r + 1 : job.last_valid) - (s & 1) * BS;
#pragma unroll
        for (int i = 0; i < BS; ++i) x[i] = (i >= limit) ? -INFINITY : x[i];
      }
      // row max over four independent chains
      float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]), m2 = fmaxf(x[4], x[5]),
            m3 = fmaxf(x[6], x[7]);
#pragma unroll
      for (int i = 8; i < BS; i += 8) {
        m0 = max3(m0, x[i], x[i + 1]);
        m1 = max3(m1, x[i + 2], x[i + 3]);
        m2 = max3(m2, x[i + 4], x[i + 5]);
        m3 = max3(m3, x[i + 6], x[i + 7]);
      }
      // A fully masked step (the second half of a diagonal tile, rows < 64) has
      // mt = -inf; it never comes first, so ms is finite by then.
      const float mt = max3(m0, m1, fmaxf(m2, m3)) * c;
      const bool need = mt > ms + kRescaleSlack;  // always on the first step (ms = -inf)
      const float m_new = need ? mt : ms;
      const float alpha = need ? ex2(ms - m_new) : 1.0f;
      const uint64_t cc = f2(c, c);
      const uint64_t mm = f2(-m_new, -m_new);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      // P in 32 packed columns; the S values are all in registers already, so P may
      // overwrite the start of its own S buffer right away.
      {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float y0, y1;
          unf2(fma2(f2(x[2 * i], x[2 * i + 1]), cc, mm), y0, y1);
          const float p0 = ex2(y0), p1 = ex2(y1);
          acc[i & 3] = add2(acc[i & 3], f2(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tSb, pk);
      }
      float s0, s1, s2, s3, s4, s5, s6, s7;
      unf2(acc[0], s0, s1);
      unf2(acc[1], s2, s3);
      unf2(acc[2], s4, s5);
      unf2(acc[3], s6, s7);
      l = l * alpha + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
      // O changes only once PV_{g-1} has finished. S_g was issued after PV_{g-2} (within
      // an item; across items after the previous item's last PV), and PV_g needs P_g,
      // so PV_{g-1} is the only product pending on o_done: an exact phase wait.
      if (s > 0 && __any_sync(0xffffffffu, need)) {
        if (!warp_wait(bar_od, (g - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
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
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_pf0 + 8 * b);
    }
    // ---------------------------------------------------------------- hand-off
    // The row's LSE goes out here; 1/l goes to the epilogue warpgroup, which
    // divides O once the item's last PV is done.
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) fail(misc, a.err_flag);
    // rows of an item that read an out-of-range table entry become NaN (only that item's)
    if (*reinterpret_cast<volatile int*>(&misc->bad_item[k % NBAD]) == id) ok = false;
    const float lse_row = ok ? (ms + log2f(l)) * kLn2F : NAN;
    if constexpr (CHUNK) {
      const int G = a.n_qo_heads / a.n_kv_heads;
      const int t = job.q0 + r / G;
      if (t < a.chunk_len && a.lse)
        a.lse[((size_t)job.b * H + job.g * G + r % G) * a.chunk_len + t] = lse_row;
    } else if constexpr (CAUSAL) {
      const int t = job.q0 + r;
      if (t < a.seq_len && a.lse) a.lse[((size_t)job.b * H + job.h) * a.seq_len + t] = lse_row;
    } else {
      const int G = a.n_qo_heads / a.n_kv_heads;
      const int req = job.r0 + r / G;
      if (req < a.n_requests)
        a.part_lse[((size_t)job.c * a.n_requests + req) * H + job.g * G + r % G] = lse_row;
    }
    if (st_cnt > 0 && ok && !warp_wait(bar_ie, (st_cnt - 1) & 1)) ok = false;
    inv_rows[r] = ok ? 1.0f / l : NAN;
    ++st_cnt;
    mbar_arrive(bar_st);
  }
}

// The epilogue warpgroup: for each item and each of its query tiles, waits for the
// tile's 1/l and its last PV, then writes O / l to global memory and frees O.
template <bool CAUSAL, bool CHUNK = false>
__device__ __forceinline__ void epilogue_loop(const TileArgs& a, Misc* misc, uint32_t (&bars)[8],
                                              const float* inv_rows_base, int n_items,
                                              const NextRing& ring, int warp, int lane) {
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
  const int H = a.n_qo_heads;
  uint32_t st_cnt[2] = {0, 0}, oi_cnt[2] = {0, 0};
  bool ok = true;
  uint32_t k = 0;
  for (int id = blockIdx.x; id < n_items; id = next_item(ring, k++, n_items, a.err_flag)) {
    const Item it = make_item<CAUSAL, CHUNK>(a, id);
    for (int t = 0; t < 2; ++t) {
      const TileJob& job = t == 0 ? it.A : it.B;
      if (job.n_tiles == 0) continue;
      const uint32_t bar_st = bars[t], bar_oi = bars[2 + t], bar_of = bars[4 + t], bar_ie = bars[6 + t];
      if (ok && !warp_wait(bar_st, st_cnt[t] & 1)) ok = false;
      ++st_cnt[t];
      // o_item has one phase per item: the next one needs this item's O freed first.
      if (ok && !warp_wait(bar_oi, oi_cnt[t] & 1)) ok = false;
      ++oi_cnt[t];
      tc_fence_after();
      if (!ok && lane == 0) fail(misc, a.err_flag);
      const float inv = ok ? inv_rows_base[t * BM + r] : NAN;
      mbar_arrive(bar_ie);  // the softmax may write this tile's next 1/l
      const uint32_t tO = misc->tmem_base + lane_addr + COL_O + t * HD;
      if constexpr (CAUSAL || CHUNK) {
        // causal: row r is token q0 + r of head h; chunk: new token q0 + r/G of query head
        // g*G + r%G. Rows past a ragged end are computed but not stored.
        const int G = a.n_qo_heads / a.n_kv_heads;
        const int tt = CHUNK ? job.q0 + r / G : job.q0 + r;
        const int hh = CHUNK ? job.g * G + r % G : job.h;
        const int T = CHUNK ? a.chunk_len : a.seq_len;
        const bool store = tt < T;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                              (((size_t)job.b * T + (store ? tt : 0)) * H + hh) * HD);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + q * 32, o);
          tmem_ld_wait();
          if (q == 3) {  // O is out of TMEM: the next item's first PV may overwrite it
            tc_fence_before();
            mbar_arrive(bar_of);
          }
          if (store) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[q * 4 + i] = make_uint4(
                  pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                  pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
          }
        }
      } else {
        const int G = a.n_qo_heads / a.n_kv_heads;
        const int req = job.r0 + r / G;
        const bool store = req < a.n_requests;
        const size_t row = ((size_t)job.c * a.n_requests + (store ? req : 0)) * H + job.g * G + r % G;
        float4* dst = reinterpret_cast<float4*>(a.part_o + row * HD);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + q * 32, o);
          tmem_ld_wait();
          if (q == 3) {
            tc_fence_before();
            mbar_arrive(bar_of);
          }
          if (store) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[q * 8 + i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                           __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
          }
        }
      }
    }
  }
}

// One CTA per item in the grid; a running CTA also takes the items of CTAs that have
// not started yet (work distribution above), so one CTA per SM runs to the end.
template <bool CAUSAL, bool CHUNK = false>
__global__ void __launch_bounds__(THREADS, 1)
attn_tile_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const TileArgs a, int n_items) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  Misc* misc = reinterpret_cast<Misc*>(smem + SM_MISC);
  auto bar = [&](int i) { return sb + SM_BAR + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.n_qo_heads / a.n_kv_heads;
  if constexpr (!CAUSAL && !CHUNK) {
    // The cascade's suffix decode, launched after this kernel on the same stream, may start
    // now: it streams its own pages and waits for this grid before reading its results.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      const bool per_thread = (i >= BAR_PF && i < BAR_PF + 4) || i == BAR_OF || i == BAR_OF + 1 ||
                              i == BAR_ST || i == BAR_ST + 1 || i == BAR_IE || i == BAR_IE + 1;
      const bool per_issuer = (i >= BAR_KE && i < BAR_KE + NSK) || (i >= BAR_VE && i < BAR_VE + NSV);
      const bool per_warp = i >= BAR_NE && i < BAR_NE + NXS;
      mbar_init(bar(i), per_thread ? 128 : (per_issuer ? 2 : (per_warp ? THREADS / 32 : 1)));
    }
    misc->abort_ = 0;
    for (int i = 0; i < NBAD; ++i) misc->bad_item[i] = -1;
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
  const NextRing ring{smem_u32(&misc->next[0]), bar(BAR_NF), bar(BAR_NE)};
  // Registers are rebalanced between warpgroups with setmaxnreg, which every warp of a
  // warpgroup executes at the same instruction. Each warpgroup's code sits in one
  // branch that starts with its setmaxnreg, so the compiler allocates that code within
  // the new limit: code the instruction does not dominate may use registers that the
  // instruction has already released.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0 || warp == 3) {
      // ------------------------------------------------------------------ TMA producers
      // Warp 0 streams Q and K tiles, warp 3 the V tiles: each waits only on its own
      // ring, so a tile's next item can start while the other tile still drains V.
      {
        if (elect_one()) {
          tma_prefetch_desc(&mq);
          tma_prefetch_desc(&mk);
          tma_prefetch_desc(&mv);
        }
        __syncwarp();
        const bool v_role = warp == 3;
        uint32_t k_cnt = 0, v_cnt = 0, q_cnt = 0;
        bool ok = true;
        uint32_t k = 0, n_req = 0;  // k: this CTA's item count, the current item's sequence number
        // One 128-key tile of K or V (32 KiB) into its ring.
        auto load_tile = [&](const Item& it, int j, bool is_v) -> bool {
          uint32_t& cnt = is_v ? v_cnt : k_cnt;
          const uint32_t ns = is_v ? NSV : NSK;
          const uint32_t s = cnt % ns, u = cnt / ns;
          const uint32_t full = bar((is_v ? BAR_VF : BAR_KF) + s);
          if (u > 0 && !warp_wait(bar((is_v ? BAR_VE : BAR_KE) + s), (u - 1) & 1)) return false;
          if (__any_sync(0xffffffffu, misc->abort_ != 0)) return false;
          const uint32_t dst = sb + (is_v ? SM_V : SM_K) + s * TILE;
          const CUtensorMap* map = is_v ? &mv : &mk;
          ++cnt;
          if (!elect_one()) {
            __syncwarp();
            return true;
          }
          if constexpr (CAUSAL) {
            mbar_arrive_expect_tx(full, TILE);
            const int k0 = j * BN;
            tma_load_4d(dst, map, 0, it.hk, k0, it.b, full);
            tma_load_4d(dst + SUB, map, 64, it.hk, k0, it.b, full);
          } else {
            // Eight pages of 16 keys make one 128-key tile; each page is a 16-row box.
            // Slots past the prefix (or the sequence) reload its first page (finite data;
            // masked out).
            // chunk: the sequence's own pages, up to its last new token
            const int n_seq_pages = CHUNK ? (it.A.L0 + a.chunk_len + 15) / 16 : a.n_prefix_pages;
            const int32_t* table = CHUNK ? a.block_table + (size_t)it.b * a.max_blocks : a.prefix_table;
            int phys[8];
            bool bad = false;
#pragma unroll
            for (int pp = 0; pp < 8; ++pp) {
              const int page_idx = (it.kv_first + j) * 8 + pp;
              phys[pp] = __ldg(table + (page_idx < n_seq_pages ? page_idx : 0));
              if (phys[pp] < 0 || phys[pp] >= a.num_pages) {
                bad = true;
                phys[pp] = 0;
              }
            }
            // The mark is written before the arrival below, which publishes it with the tile.
            if (bad) {
              misc->bad_item[k % NBAD] = it.id;
              set_err(a.err_flag, PKV_DEVERR_BAD_PAGE);
            }
            mbar_arrive_expect_tx(full, TILE);
#pragma unroll
            for (int pp = 0; pp < 8; ++pp) {
              const int row = (phys[pp] * a.n_kv_heads + it.hk) * 16;
              tma_load_2d(dst + pp * 2048, map, 0, row, full);
              tma_load_2d(dst + SUB + pp * 2048, map, 64, row, full);
            }
          }
          __syncwarp();
          return true;
        };
        for (int id = blockIdx.x; ok && id < n_items; id = next_item(ring, k++, n_items, a.err_flag)) {
          const Item it = make_item<CAUSAL, CHUNK>(a, id);
          // Q tile n = 2k + t goes to buffer n % NQ once the products of Q tile n - NQ (the
          // last one in that buffer) are done.
          auto load_q = [&](int t) -> bool {
            const uint32_t n = q_cnt;
            const uint32_t qf = bar(BAR_QF + n % NQB);
            if (n >= NQ && !warp_wait(bar(BAR_QE + (n - NQ) % NQB), ((n - NQ) / NQB) & 1)) return false;
            ++q_cnt;
            if (elect_one()) {
              mbar_arrive_expect_tx(qf, TILE);
              for (int half = 0; half < 2; ++half) {
                const uint32_t dst = sb + SM_Q + (n % NQ) * TILE + half * SUB;
                if constexpr (CHUNK)
                  tma_load_4d(dst, &mq, half * 64, it.hk * G, (t == 0 ? it.A : it.B).q0, it.b, qf);
                else if constexpr (CAUSAL)
                  tma_load_4d(dst, &mq, half * 64, it.A.h, it.qrow + t * BM, it.b, qf);
                else
                  tma_load_3d(dst, &mq, half * 64, it.hk * G, (it.qrow + t * BM) / G, qf);
              }
            }
            __syncwarp();
            return true;
          };
          if (v_role) {
            for (int j = 0; ok && j < it.n_kv; ++j) ok = load_tile(it, j, true);
          } else {
            // Q_A, K0, Q_B, K1, K2, ...: both tiles can start as soon as K0 is in.
            // Ask for the next item just before this one's last kReqAhead K tiles: the
            // response (which takes about a microsecond) is back by the time tile A could
            // start the next item, and the CTA holds the next item for as short a time as
            // that allows.
            auto request = [&]() {
              const uint32_t s = k % NXS, u = k / NXS;
              if (ok && u > 0 && !warp_wait(ring.empty0 + 8 * s, (u - 1) & 1)) ok = false;
              if (ok) {
                if (elect_one()) request_next_cta(ring.slot0 + 16 * s, ring.full0 + 8 * s);
                __syncwarp();
                ++n_req;
              }
            };
            ok = load_q(0) && load_tile(it, 0, false) && load_q(1);
            const int j_req = it.n_kv - kReqAhead;
            bool asked = false;
            for (int j = 1; ok && j < it.n_kv; ++j) {
              if (j == j_req) {
                request();
                asked = true;
              }
              ok = ok && load_tile(it, j, false);
            }
            if (!asked) request();
          }
        }
        // A request still in flight must land before the CTA's shared memory is released.
        if (!v_role && n_req > k && !warp_wait(ring.full0 + 8 * ((n_req - 1) % NXS), ((n_req - 1) / NXS) & 1) &&
            lane == 0)
          set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
        if (!ok && lane == 0) fail(misc, a.err_flag);
        // Every issued copy must land before the CTA's shared memory is released
        // (immediate on the normal path, where the MMA warp already waited for them).
        bool drained = true;
        for (uint32_t n = q_cnt > NQB ? q_cnt - NQB : 0; n < q_cnt; ++n)
          if (!warp_wait(bar(BAR_QF + n % NQB), (n / NQB) & 1)) drained = false;
        for (uint32_t s = 0; s < NSK && s < k_cnt; ++s)
          if (!warp_wait(bar(BAR_KF + s), ((k_cnt - 1 - s) / NSK) & 1)) drained = false;
        for (uint32_t s = 0; s < NSV && s < v_cnt; ++s)
          if (!warp_wait(bar(BAR_VF + s), ((v_cnt - 1 - s) / NSV) & 1)) drained = false;
        if (!drained && lane == 0) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
      }
    } else if (warp == 1 || warp == 2) {
      // ------------------------------------------------------------------ MMA issuers
      // One thread per query tile (warp 1: A, warp 2: B), so each tile's chain
      // S -> softmax -> PV runs at its own pace, and tile A moves on to the next item
      // while B finishes. They share only the K/V stages, whose release barriers take
      // one arrival from each.
      {
        const int t = warp - 1;
        const uint32_t idS = idesc_bf16_f32(BM, BS, false, false);
        const uint32_t idPV = idesc_bf16_f32(BM, HD, false, true);
        // Descriptors are built once; a K step inside a tile only moves the start
        // address, i.e. adds (byte offset >> 4) to the low field. The largest start
        // (under 232 KB) plus the largest step stays inside the 14-bit field. Ring slots
        // and the two Q tiles are TILE bytes apart: slot i's descriptor is the first
        // slot's plus i * (TILE >> 4).
        constexpr uint64_t kSlot = TILE >> 4;
        const uint64_t dq0 = smem_desc(sb + SM_Q, 16, 1024, kSwizzle128B);
        const uint64_t dk0 = smem_desc(sb + SM_K, 16, 1024, kSwizzle128B);
        const uint64_t dv0 = smem_desc(sb + SM_V, 16384, 1024, kSwizzle128B);
        const uint32_t d_s = tmem + COL_S + t * BN, d_o = tmem + COL_O + t * HD;
        // S for global step gs (keys [64*half, 64*half + 64) of the K tile at ring position
        // kg) into S buffer gs & 1; then the K stage's release (rel arrivals) after the
        // tile's second half, and Q_t's release after the item's last step.
        auto issue_s = [&](uint32_t gs, uint32_t kg, uint64_t dq, int half, int rel_n, uint32_t q_empty) {
          const uint64_t b0 = dk0 + (uint64_t)(kg % NSK) * kSlot + (uint64_t)((half * BS * 128) >> 4);
          if (elect_one()) {
  #pragma unroll
            for (int k = 0; k < HD / 16; ++k) {
              const uint64_t off = (uint64_t)(((k / 4) * SUB + (k % 4) * 32) >> 4);
              mma_bf16_ss(d_s + (gs & 1) * BS, dq + off, b0 + off, idS, k > 0);
            }
            mma_commit(bar(BAR_SF + 2 * t + (gs & 1)));
            if (q_empty) mma_commit(q_empty);  // the last product that reads this Q tile
            for (int i = 0; i < rel_n; ++i) mma_commit(bar(BAR_KE + kg % NSK));
          }
          __syncwarp();
        };
        // O_t (+)= P_gp V over keys [64*half, +64) of the V tile at ring position vg; then
        // o_done, the V stage's release after the tile's second half, o_item after the
        // item's last step.
        auto issue_pv = [&](uint32_t gp, uint32_t vg, int half, bool first, int rel_n, bool last) {
          const uint64_t b0 = dv0 + (uint64_t)(vg % NSV) * kSlot;
          if (elect_one()) {
  #pragma unroll
            for (int k = 0; k < BS / 16; ++k)
              mma_bf16_ts(d_o, d_s + (gp & 1) * BS + k * 8, b0 + (uint64_t)(((half * 4 + k) * 2048) >> 4),
                          idPV, (!first || k > 0) ? 1u : 0u);
            mma_commit(bar(BAR_OD + t));
            for (int i = 0; i < rel_n; ++i) mma_commit(bar(BAR_VE + vg % NSV));
            if (last) mma_commit(bar(BAR_OI + t));
          }
          __syncwarp();
        };
        uint32_t k_cnt = 0, v_cnt = 0, g = 0, of_cnt = 0, of_need = 0, vz_cnt = 0;
        bool ok = true;
        uint32_t k = 0;
        for (int id = blockIdx.x; ok && id < n_items; id = next_item(ring, k++, n_items, a.err_flag)) {
          const Item it = make_item<CAUSAL, CHUNK>(a, id);
          const int n_t = (t == 0 ? it.A : it.B).n_tiles;  // key tiles this tile reads
          const int n_o = (t == 0 ? it.B : it.A).n_tiles;  // key tiles the other tile reads
          const int n_kv = it.n_kv;
          // Only an issuer that reads a stage releases it. Where the other tile does not
          // read stage j (j >= n_o), this issuer brings both arrivals, so a stage is never
          // handed back to TMA while a product of either tile may still read it.
          auto rel = [&](int j) { return j < n_o ? 1 : 2; };
          // This item's Q tile n = 2k + t: buffer n % NQ, barriers n % NQB.
          const uint32_t qn = 2 * k + t;
          const uint32_t q_full = bar(BAR_QF + qn % NQB), q_empty = bar(BAR_QE + qn % NQB);
          const uint64_t dq = dq0 + (uint64_t)(qn % NQ) * kSlot;
          if (!warp_wait(q_full, (qn / NQB) & 1)) {
            ok = false;
            break;
          }
          if (n_t == 0) {  // only B can be missing: A covers the K/V arrivals
            if (elect_one()) mma_commit(q_empty);  // its Q_B (never read) may be replaced
            __syncwarp();
            k_cnt += n_kv;
            v_cnt += n_kv;
            continue;
          }
          const int n_s = 2 * n_t;  // 64-key steps
          if (!warp_wait(bar(BAR_KF + k_cnt % NSK), (k_cnt / NSK) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // S for the first two steps (both halves of K tile 0); the buffers were last read
          // by the previous item's last two PV products, issued earlier by this thread.
          issue_s(g, k_cnt, dq, 0, 0, 0);
          issue_s(g + 1, k_cnt, dq, 1, rel(0), n_s == 2 ? q_empty : 0);
          for (int st = 0; st < n_s; ++st, ++g) {
            const int j = st >> 1, half = st & 1;
            if (!warp_wait(bar(BAR_PF + 2 * t + (g & 1)), (g >> 1) & 1)) { ok = false; break; }
            // the previous item's epilogue must have read O before it is overwritten
            if (st == 0 && of_need > of_cnt) {
              if (!warp_wait(bar(BAR_OF + t), of_cnt & 1)) { ok = false; break; }
              ++of_cnt;
            }
            const uint32_t vg = v_cnt + j;
            if (half == 0 && !warp_wait(bar(BAR_VF + vg % NSV), (vg / NSV) & 1)) { ok = false; break; }
            if constexpr (CHUNK) {
              // The tile holding the sequence's last key also holds page slots past it,
              // whose contents are not the caller's data (they may not even be finite): zero
              // those V rows, since a masked key still enters PV as 0 x V. One issuer zeroes
              // them: B's when both tiles read that key tile (B's key range contains A's),
              // and A waits for it before its product; the writes are made visible to the
              // tensor core first.
              const int pos_end = it.A.L0 + a.chunk_len;  // keys [0, pos_end) exist
              const int j_last = (pos_end - 1) / BN;
              if (half == 0 && j == j_last) {
                const bool b_reads = it.B.n_tiles > 0 && it.B.n_tiles - 1 == j_last;
                const bool a_reads = it.A.n_tiles - 1 == j_last;
                if (t == 1 || !b_reads) {
                  unsigned char* vt = smem + SM_V + (vg % NSV) * TILE;
                  for (int row = pos_end - j * BN + (lane >> 3); row < BN; row += 4)
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub)
                      *reinterpret_cast<uint4*>(vt + sub * SUB + row * 128 + (lane & 7) * 16) =
                          make_uint4(0u, 0u, 0u, 0u);
                  fence_proxy_async_smem();
                  __syncwarp();
                  if (t == 1 && a_reads) {
                    if (elect_one()) mbar_arrive(bar(BAR_VZ));
                    __syncwarp();
                  }
                } else {
                  if (!warp_wait(bar(BAR_VZ), vz_cnt & 1)) { ok = false; break; }
                  ++vz_cnt;
                }
              }
            }
            tc_fence_after();
            issue_pv(g, vg, half, st == 0, half == 1 ? rel(j) : 0, st == n_s - 1);
            // S two steps ahead reuses P_g's buffer: the in-order tensor pipe reads P_g first.
            const int sn = st + 2;
            if (sn < n_s) {
              const uint32_t kg = k_cnt + (sn >> 1);
              if ((sn & 1) == 0 && !warp_wait(bar(BAR_KF + kg % NSK), (kg / NSK) & 1)) { ok = false; break; }
              tc_fence_after();
              issue_s(g + 2, kg, dq, sn & 1, (sn & 1) ? rel(sn >> 1) : 0, sn == n_s - 1 ? q_empty : 0);
            }
          }
          k_cnt += n_kv;
          v_cnt += n_kv;
          ++of_need;
        }
        if (!ok && lane == 0) fail(misc, a.err_flag);
        // Every issued product must finish before TMEM is freed.
        if (elect_one()) mma_commit(bar(BAR_DRAIN + t));
        __syncwarp();
        if (!warp_wait(bar(BAR_DRAIN + t), 0) && lane == 0) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
      }
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
    const int t = (warp - 4) / 4;
    softmax_loop<CAUSAL, CHUNK>(a, misc, bar(BAR_SF + 2 * t), bar(BAR_PF + 2 * t), bar(BAR_OD + t),
                         bar(BAR_ST + t), bar(BAR_IE + t),
                         reinterpret_cast<float*>(smem + SM_INV) + t * BM, COL_S + t * BN,
                         COL_O + t * HD, t, n_items, ring, warp, lane);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    uint32_t bars[8] = {bar(BAR_ST), bar(BAR_ST + 1), bar(BAR_OI),     bar(BAR_OI + 1),
                        bar(BAR_OF), bar(BAR_OF + 1), bar(BAR_IE), bar(BAR_IE + 1)};
    epilogue_loop<CAUSAL, CHUNK>(a, misc, bars, reinterpret_cast<const float*>(smem + SM_INV), n_items, ring,
                          warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Resolved once per process (a function-local static is initialised by one thread only).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
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

template <bool CAUSAL, bool CHUNK = false>
int launch_tiles(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                 const TileArgs& a, long n_items, cudaStream_t stream) {
  if (n_items <= 0) return PKV_OK;
  if (n_items > 0x7fffffffL) return PKV_ERR_UNSUPPORTED;
  static FuncConfigured configured;
  if (!configured.ensure(reinterpret_cast<const void*>(attn_tile_kernel<CAUSAL, CHUNK>), SMEM_BYTES))
    return PKV_ERR_LAUNCH;
  // One CTA per item: the CTAs that run first take over the rest (work distribution).
  attn_tile_kernel<CAUSAL, CHUNK><<<(unsigned)n_items, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, a,
                                                                                  (int)n_items);
  return check_launch(cudaGetLastError());
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return encode_fn(); }

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
  // About 64 items per group, and a tail of about 1.25 waves of items (measured on the
  // batch-8, T-1024, 32-head workload: groups of 16 (b, h) and a 48-(b, h) tail gave
  // about 880 TFLOP/s, against about 855 for groups of 32 without a tail, 813 for
  // longest first throughout and about 795 for a static round-robin over persistent CTAs).
  const int n_pairs = (int)((n_qt + 1) / 2);
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  a.group_bh = 64 / n_pairs > 1 ? 64 / n_pairs : 1;
  a.tail_bh = (5 * sms / 4 + n_pairs - 1) / n_pairs;
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

// Chunked prefill over the paged cache: the non-causal tile kernel's third mode. A query
// tile is 128/G new tokens x the G query heads of one KV head (as in the prefix mode), K/V
// are gathered page by page through each sequence's own block table, and row r of a tile
// sees the keys up to its own position prefix_len + token.
int launch_prefill_chunk(const ChunkArgs& c, cudaStream_t stream) {
  if (c.head_dim != HD || c.page_size != 16) return PKV_ERR_UNSUPPORTED;
  const int G = c.n_qo_heads / c.n_kv_heads;
  if (BM % G) return PKV_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  {
    // q [B, C, Hq, D] as (D, Hq, C, B): one box = G heads x 128/G tokens = 128 rows of 64
    cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)c.n_qo_heads, (cuuint64_t)c.chunk_len,
                          (cuuint64_t)c.batch};
    cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)c.n_qo_heads * HD * 2,
                             (cuuint64_t)c.chunk_len * c.n_qo_heads * HD * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(BM / G), 1};
    if (!encode(&mq, c.q, 4, dims, strides, box)) return check_launch(cudaErrorInvalidValue);
  }
  {
    // pools [pages, Hkv, 16, D] as rows of D: one box = one (page, head) tile, 16 rows x 64
    const cuuint64_t rows = (cuuint64_t)c.num_pages * c.n_kv_heads * 16;
    cuuint64_t dims[2] = {(cuuint64_t)HD, rows};
    cuuint64_t strides[1] = {(cuuint64_t)HD * 2};
    cuuint32_t box[2] = {64, 16};
    if (!encode(&mk, c.k_pages, 2, dims, strides, box) || !encode(&mv, c.v_pages, 2, dims, strides, box))
      return check_launch(cudaErrorInvalidValue);
  }
  TileArgs a{};
  a.out = c.out;
  a.lse = c.lse;
  a.err_flag = c.err_flag;
  a.scale = c.scale;
  a.batch = c.batch;
  a.n_qo_heads = c.n_qo_heads;
  a.n_kv_heads = c.n_kv_heads;
  a.num_pages = c.num_pages;
  a.block_table = c.block_table;
  a.prefix_lens = c.prefix_lens;
  a.chunk_len = c.chunk_len;
  a.max_blocks = c.max_blocks;
  const long tpt = BM / G;
  const long n_qt = (c.chunk_len + tpt - 1) / tpt;
  const long grid = (n_qt + 1) / 2 * c.n_kv_heads * c.batch;
  // The same grouping as the causal prefill: about 64 items per group, a tail of about 1.25
  // waves of items. Without it the pairs of one (sequence, KV head) ran a wave or more apart
  // and each re-read the sequence's K/V from DRAM (about 3.7x the algorithmic bytes).
  const int n_pairs = (int)((n_qt + 1) / 2);
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  a.group_bh = 64 / n_pairs > 1 ? 64 / n_pairs : 1;
  a.tail_bh = (5 * sms / 4 + n_pairs - 1) / n_pairs;
  return launch_tiles<false, true>(mq, mk, mv, a, grid, stream);
}

}  // namespace pkv
