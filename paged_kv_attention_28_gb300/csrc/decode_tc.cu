// Paged decode for GQA groups of 4 or 8 query heads on the sm_103a tensor cores.
//
// With G query heads per KV head, every key and value element of the cache takes part
// in G dot-product terms and G weighted sums. At HBM speed that is, for G = 8, about
// 110 TFLOP/s of multiply-adds: more than the fp32 CUDA cores deliver, so on CUDA cores
// a GQA decode is bound by its arithmetic, not by its bytes. Here both products of the
// online softmax ("快速注意力内核与算子融合", Q&A on FlashAttention tiling; partial states
// per split as in "【FlashAttention-V4，非官方】FlashDecoding++", section 1) run on tcgen05,
// with the keys as the 128-row operand:
//   S^T [128 keys x 16]  = K_tile [128 keys x 128 dims]  . Q^T [128 dims x 16 heads]
//   O^T [128 dims x 16] += V_tile^T [128 dims x 128 keys] . P^T [128 keys x 16 heads]
// The group's heads are the products' N = 16 (rows past G are padding). A tile is 128
// keys = 8 pages of 16, gathered through the block table ("快速注意力内核与算子融合", Q&A on
// paged attention) by 2-D TMA boxes of one (page, KV head) half-row block each.
//
// Work: a unit is (split, KV head, sequence), as for the CUDA-core decode, and writes the
// same outputs (the final row, or an fp32 partial state for the split merge). The grid
// has one CTA per unit and one CTA fits on an SM; a running CTA takes the pending units
// (work_queue.cuh), so the rings and TMEM stay warm from one unit to the next.
//
// With one split per sequence the units' lengths differ as the sequences do; every CTA then
// ranks the sequences by length (a counting sort over 128-key tiles) and hands out the
// longest first, so that the last units to start are short ones.
//
// Warps (352 threads): warp 0 TMA producer of Q and K tiles (and TMEM owner), warp 1 MMA
// issuer, warp 2 TMA producer of V tiles, warps 3..6 the softmax: thread t of those 128
// owns key t of a tile (TMEM lane t); warps 7..10 the epilogue: thread t owns head-dim t
// of O. Warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31.
// TMEM: S^T double-buffered (columns 0..15 and 16..31), O^T double-buffered by unit
// (columns 32..47 and 48..63).
// Shared memory: K and V rings of 3 tiles (32 KiB each), Q and P^T double-buffered (4 KiB
// each), a small reduction area, the barriers, the sequence order.
//
// E4M3 pools (groups of 4 and 8): the producers copy tiles of codes into staging rings; warps
// 11 .. 16 (544 threads) convert them to f16 into K and V rings of 2 tiles, and the products
// take f16 operands (see produce_fp8 and convert_fp8).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "internal.h"
#include "tcgen05.cuh"
#include "work_queue.cuh"

namespace pkv {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();  // prefill.cu

namespace {

constexpr int TK = 128;                  // keys per tile
constexpr int TD = 128;                  // head dim
constexpr int NQ = 16;                   // N of both products: the group, padded
constexpr int KVT = TK * TD * 2;         // one K or V tile: 32 KiB
constexpr int KVH = KVT / 2;             // one 64-column half of it: [128 rows][128 bytes]
constexpr int QB = NQ * TD * 2;          // Q tile: 4 KiB, two halves of [16 rows][128 bytes]
constexpr int PB = NQ * TK * 2;          // one P^T buffer: 4 KiB, two 64-key halves
constexpr int NRED = 5;                  // reduction buffers: per step (2), final sums, fallback maxima (2)
// barriers (one per stage or buffer): k_full k_empty v_full v_empty (3 each), q_full q_empty,
// s_full s_empty, p_full p_empty (2 each), o_done, u_done o_free st_full st_empty (2 each, by
// unit parity), drain, next_full next_empty (4 each), red (5: a reduction's parts are in);
// E4M3 pools only: k_landed v_landed (a staging tile's copies are in, 3 each), q_conv (2: the
// unit's q is in f16), k_staged_free v_staged_free (the converters have read a staging tile, 3
// each)
constexpr int B_KF = 0, B_KE = 3, B_VF = 6, B_VE = 9, B_QF = 12, B_QE = 14, B_SF = 16, B_SE = 18,
              B_PF = 20, B_PE = 22, B_OD = 24, B_UD = 25, B_OF = 27, B_STF = 29, B_STE = 31, B_DR = 33,
              B_NF = 34, B_NE = 38, B_RED = 42, B_KT = 47, B_VT = 50, B_QC = 53, B_KSE = 55, B_VSE = 58,
              NBAR = 64;
constexpr int LPT_MAX = 2048;            // longest-first order for batches up to this size
constexpr int LPT_BUCKETS = 64;          // by 128-key tiles; 63 or more share the first bucket
static_assert(LPT_BUCKETS == 64 && LPT_MAX <= 65536, "the order's scan and index type");

// Shared-memory layout. bf16 pools: K and V rings of 3 tiles. E4M3 pools: K and V rings of 2
// f16 tiles, each fed from a staging ring of 2 tiles of codes (16 KiB) that the copies fill.
template <bool FP8>
struct TcL {
  // E4M3 pools: warps 11 .. 13 convert K tiles, 14 .. 16 V tiles
  static constexpr int NCV = 3;                                // converter warps per ring
  static constexpr int THREADS = FP8 ? 352 + 2 * NCV * 32 : 352;
  static constexpr int NWARP = THREADS / 32;
  static constexpr int NSK = FP8 ? 2 : 3, NSV = FP8 ? 2 : 3;  // ring stages
  static constexpr int NSTG = FP8 ? 2 : 0;                    // staging tiles per ring
  static constexpr int STG = TK * TD;                          // one staging tile of codes
  static constexpr int SM_K = 0;
  static constexpr int SM_V = SM_K + NSK * KVT;
  static constexpr int SM_KS = SM_V + NSV * KVT;
  static constexpr int SM_VS = SM_KS + NSTG * STG;
  static constexpr int SM_Q = SM_VS + NSTG * STG;  // Q double-buffered by unit
  static constexpr int SM_P = SM_Q + 2 * QB;
  static constexpr int SM_RED = SM_P + 2 * PB;     // float [NRED][4 warps][NQ]
  static constexpr int SM_ST = SM_RED + NRED * 4 * NQ * 4;  // float [2 units][NQ][2]: each head's (max, sum)
  static constexpr int SM_BAR = SM_ST + 2 * NQ * 2 * 4;
  static constexpr int SM_SC = SM_BAR + NBAR * 8;  // float [3 V stages][8 pages][2]: (K, V) scales
  static constexpr int SM_QU = SM_SC + 3 * 8 * 2 * 4;  // float [2 units][NQ]: each q row's 2^-sh
  static constexpr int SM_PH = SM_QU + 2 * NQ * 4;      // int [K, V][3 staging slots][8]: the tiles' pages
  static constexpr int SM_MISC = SM_PH + 2 * 3 * 8 * 4;
  static constexpr int SM_HIST = SM_MISC + 128;    // int [LPT_BUCKETS]
  static constexpr int SM_ORD = SM_HIST + LPT_BUCKETS * 4;  // uint16 [LPT_MAX]: sequences, longest first
  static constexpr int SM_BK = SM_ORD + LPT_MAX * 2;        // uint8 [LPT_MAX]: each sequence's bucket
  static constexpr int SMEM = SM_BK + LPT_MAX + 1024;       // + slack to align the base to 1024
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(SM_MISC % 16 == 0 && SM_Q % 1024 == 0 && SM_P % 1024 == 0 && SM_KS % 1024 == 0 &&
                    SM_VS % 1024 == 0,
                "layout");
  static_assert(NSK <= 3 && NSV <= 3 && NSTG <= 3, "barrier slots");
};
constexpr int TMEM_COLS = 64;
constexpr int COL_S = 0, COL_O = 32;  // S^T buffers at 0 and 16, O^T buffers at 32 and 48
constexpr float kL2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.0f;  // lazy rescale: a head's reference max moves when a tile beats it by 8 (log2)
constexpr int NBADM = 8;
constexpr float kUnifiedBetaTc = 60.0f;  // unified-max margin, natural-log units (as in the CUDA-core kernel)

struct Misc {
  uint4 next[NXS];
  uint32_t tmem_base;
  int abort_;
  int bad_item[NBADM];  // as in the tile kernel: the id of this CTA's k-th unit if it met a bad page
};
static_assert(sizeof(Misc) <= 128, "Misc");

// One unit: where its keys are and where its rows go.
struct Unit {
  int split, hk, b;
  int first, n_pages, kv_len;  // the split's first page (index into the sequence's table) and count
  int n_tiles;                 // 128-key tiles (0: nothing to stream)
  int n_live;                  // splits of the sequence that hold keys
  int kind;                    // 0: stream; 1: write NaN (bad length); 2: write 0 / -inf (empty); 3: nothing
  bool final_write;            // the sequence has one live split: write out / lse directly
};

// A sequence's place in the longest-first order: its 128-key tiles, most first; a length
// the table cannot hold makes a unit that only writes NaN, so it goes last.
__device__ __forceinline__ int lpt_bucket(const DecodeArgs& a, int b) {
  const int len = __ldg(a.kv_lens + b);
  if (len < 0 || len > a.max_blocks * 16) return LPT_BUCKETS - 1;
  return LPT_BUCKETS - 1 - min((len + TK - 1) / TK, LPT_BUCKETS - 1);
}

// `ord`: the sequences in the order their units are handed out, or null for batch order.
__device__ __forceinline__ Unit make_unit(const DecodeArgs& a, int id, const uint16_t* ord) {
  Unit u{};
  u.split = id % a.num_splits;
  const int rest = id / a.num_splits;
  u.hk = rest % a.n_kv_heads;
  u.b = rest / a.n_kv_heads;
  if (ord) u.b = ord[u.b];
  u.kv_len = __ldg(a.kv_lens + u.b);
  if (u.kv_len < 0 || u.kv_len > a.max_blocks * 16) {
    u.kind = (u.split == 0 && !a.partial_only) ? 1 : 3;
    return u;
  }
  const int nblk = (u.kv_len + 15) / 16;
  const int n_live = (nblk + a.pages_per_split - 1) / a.pages_per_split;
  if (n_live == 0) {
    u.kind = (u.split == 0 && !a.partial_only) ? 2 : 3;
    return u;
  }
  if (u.split >= n_live) {
    u.kind = 3;
    return u;
  }
  u.n_live = n_live;
  u.first = u.split * a.pages_per_split;
  u.n_pages = min(a.pages_per_split, nblk - u.first);
  u.n_tiles = (u.n_pages + 7) / 8;
  u.final_write = n_live == 1 && !a.partial_only;
  return u;
}

// Keys of tile j that exist (the rest of the tile is masked).
__device__ __forceinline__ int tile_valid(const Unit& u, int j) {
  const int pages = min(8, u.n_pages - 8 * j);
  return min(pages * 16, u.kv_len - (u.first + 8 * j) * 16);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}

// Sum (or max) of x over the 128 softmax threads, for G heads: warp shuffles, then the four
// warps' values through shared memory buffer `sel`, published by an mbarrier (four
// arrivals; `phase` counts the buffer's uses) whose wait is bounded like every other.
// Returns false if the wait gave up. A buffer is written again only two uses later, once
// every warp has passed the use in between, i.e. has read it.
template <int G, bool MAX>
__device__ __forceinline__ bool block_reduce(float (&x)[G], float* red, int sel, uint32_t bar, uint32_t phase,
                                             int wq, int lane, uint64_t lim) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x[h], off);
      x[h] = MAX ? fmaxf(x[h], y) : x[h] + y;
    }
  }
  float* r = red + sel * 4 * NQ;
  if (lane < G) {
    float v = x[0];
#pragma unroll
    for (int h = 1; h < G; ++h) v = (lane == h) ? x[h] : v;
    r[wq * NQ + lane] = v;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  if (!warp_wait(bar, phase & 1, lim)) return false;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float a0 = r[h], a1 = r[NQ + h], a2 = r[2 * NQ + h], a3 = r[3 * NQ + h];
    x[h] = MAX ? fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) : (a0 + a1) + (a2 + a3);
  }
  return true;
}

// The bitwise OR of w over the 128 softmax threads (same exchange as block_reduce).
__device__ __forceinline__ bool block_or(uint32_t& w, float* red, int sel, uint32_t bar, uint32_t phase, int wq,
                                         int lane, uint64_t lim) {
  w = __reduce_or_sync(0xffffffffu, w);
  uint32_t* r = reinterpret_cast<uint32_t*>(red + sel * 4 * NQ);
  if (lane == 0) r[wq] = w;
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  if (!warp_wait(bar, phase & 1, lim)) return false;
  w = (r[0] | r[1]) | (r[2] | r[3]);
  return true;
}

// Cascade: head dim t of the G rows of a request's KV head group (rows row0 .. row0 + G - 1):
// the shared prefix's chunk states are merged by log-sum-exp with the suffix's own (val,
// lse in natural-log units; lse = -inf for no suffix keys), as the split merge does, and a
// NaN state makes the row NaN. The chunks' values of all G rows are loaded 32 / G chunks at a
// time, every load of a batch in flight before any is used.
template <int G>
__device__ __forceinline__ void cascade_merge_group(const DecodeArgs& a, size_t row0, int t, float (&val)[G],
                                                    float (&lse)[G]) {
  constexpr int CB = 32 / G;  // chunks per batch
  const size_t stride = (size_t)a.batch * a.n_qo_heads;  // rows per chunk
  float M[G], l[G], acc[G];
  bool nan[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    nan[h] = lse[h] != lse[h];
    M[h] = lse[h];
    l[h] = lse[h] == -INFINITY ? 0.0f : 1.0f;
    acc[h] = lse[h] == -INFINITY ? 0.0f : val[h];
  }
  for (int c0 = 0; c0 < a.pre_n; c0 += CB) {
    float L[G][CB], O[G][CB];
#pragma unroll
    for (int i = 0; i < CB; ++i)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const int c = c0 + i;
        const size_t r = (size_t)c * stride + row0 + h;
        L[h][i] = c < a.pre_n ? __ldcg(a.pre_lse + r) : -INFINITY;
        O[h][i] = c < a.pre_n ? __ldcg(a.pre_o + r * TD + t) : 0.0f;
      }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float Mn = M[h];
#pragma unroll
      for (int i = 0; i < CB; ++i) {
        nan[h] |= L[h][i] != L[h][i];
        Mn = fmaxf(Mn, L[h][i]);
      }
      if (Mn == -INFINITY) continue;
      const float sc = ex2((M[h] - Mn) * kL2e);  // 0 while M = -inf
      l[h] *= sc;
      acc[h] *= sc;
#pragma unroll
      for (int i = 0; i < CB; ++i) {
        const float w = ex2((L[h][i] - Mn) * kL2e);
        l[h] += w;
        acc[h] = fmaf(w, O[h][i], acc[h]);
      }
      M[h] = Mn;
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (nan[h]) {
      val[h] = NAN;
      lse[h] = NAN;
    } else if (M[h] == -INFINITY) {
      val[h] = 0.0f;
      lse[h] = -INFINITY;
    } else {
      val[h] = acc[h] / l[h];
      lse[h] = M[h] + logf(l[h]);
    }
  }
}

// Two E4M3 codes (element 2i in the low byte) to an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(pair & 0xffffu)));
  return r;
}

// The producers of the E4M3 instantiation: warp 0 copies each unit's q (bf16) and its K tiles
// of codes, warp 2 its V tiles, into staging slots (a tile is 8 pages x 16 rows x 128 codes);
// a slot is reused once the converter warps have read it. The tile's pages go to shared memory
// beside the slot, for the V converters (the page scales).
template <int G>
__device__ __forceinline__ void produce_fp8(const DecodeArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                                            const CUtensorMap& mv, unsigned char* smem, uint32_t sb, Misc* misc,
                                            const NextRing& ring, const uint16_t* ord, int n_units, int warp,
                                            int lane) {
  using L = TcL<true>;
  auto bar = [&](int i) { return sb + L::SM_BAR + 8 * i; };
  const uint64_t lim = a.wait_limit_ns;
  const bool v_role = warp == 2;
  if (elect_one()) {
    tma_prefetch_desc(v_role ? &mv : &mk);
    if (!v_role) tma_prefetch_desc(&mq);
  }
  __syncwarp();
  const int land0 = v_role ? B_VT : B_KT, sfree0 = v_role ? B_VSE : B_KSE;
  const uint32_t stg_base = v_role ? L::SM_VS : L::SM_KS;
  const CUtensorMap* map = v_role ? &mv : &mk;
  int* pages_s = reinterpret_cast<int*>(smem + L::SM_PH) + (v_role ? 3 * 8 : 0);
  uint32_t cnt = 0, qi = 0, k = 0, n_req = 0;
  bool ok = true;
  for (int id = blockIdx.x; ok && id < n_units; id = next_item(ring, k++, n_units, a.err_flag)) {
    const Unit u = make_unit(a, id, ord);
    if (u.kind == 0 && !v_role) {
      const uint32_t qb = qi & 1;
      if (qi >= 2 && !warp_wait(bar(B_QE + qb), ((qi >> 1) - 1) & 1, lim)) ok = false;
      if (ok && elect_one()) {
        mbar_arrive_expect_tx(bar(B_QF + qb), QB);
        tma_load_3d(sb + L::SM_Q + qb * QB, &mq, 0, u.hk * G, u.b, bar(B_QF + qb));
        tma_load_3d(sb + L::SM_Q + qb * QB + QB / 2, &mq, 64, u.hk * G, u.b, bar(B_QF + qb));
      }
      __syncwarp();
    }
    if (u.kind == 0) ++qi;
    if (!v_role && ok) {
      // ask for the next unit as soon as this one is known
      const uint32_t s = k % NXS, uu = k / NXS;
      if (uu > 0 && !warp_wait(ring.empty0 + 8 * s, (uu - 1) & 1, lim)) ok = false;
      if (ok) {
        if (elect_one()) request_next_cta(ring.slot0 + 16 * s, ring.full0 + 8 * s);
        __syncwarp();
        ++n_req;
      }
    }
    const int32_t* trow = a.block_table + (size_t)u.b * a.max_blocks + u.first;
    int ent = 0;
    for (int j = 0; ok && j < u.n_tiles; ++j, ++cnt) {
      if ((j & 3) == 0) ent = (32 * (j >> 2) + lane < u.n_pages) ? __ldg(trow + 32 * (j >> 2) + lane) : 0;
      const uint32_t slot = cnt % L::NSTG, use = cnt / L::NSTG;
      if (use > 0 && !warp_wait(bar(sfree0 + slot), (use - 1) & 1, lim)) {
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, misc->abort_ != 0)) {
        ok = false;
        break;
      }
      const int pages = min(8, u.n_pages - 8 * j);
      // (both shuffles are taken by the whole warp)
      const int own = __shfl_sync(0xffffffffu, ent, (8 * j + (lane & 7)) & 31);
      const int tile_first = __shfl_sync(0xffffffffu, ent, (8 * j) & 31);
      int phys = lane < pages ? own : tile_first;
      bool bad = false;
      if (lane < 8) {
        bad = phys < 0 || phys >= a.num_pages;
        if (bad) phys = 0;
        pages_s[slot * 8 + lane] = phys;  // published by the arrival below
      }
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (any_bad && lane == 0) {
        misc->bad_item[k % NBADM] = id;  // written before the arrival that publishes the tile
        set_err(a.err_flag, PKV_DEVERR_BAD_PAGE);
      }
      const bool stall = !v_role && a.stall_page >= 8 * j && a.stall_page < 8 * j + 8;
      __syncwarp();
      if (lane == 0 && !stall) mbar_arrive_expect_tx(bar(land0 + slot), L::STG);
      __syncwarp();
      if (lane < 8 && !stall)
        tma_load_2d(sb + stg_base + slot * L::STG + lane * 2048, map, 0, (phys * a.n_kv_heads + u.hk) * 16,
                    bar(land0 + slot));
      __syncwarp();
    }
  }
  if (!v_role && n_req > k && !warp_wait(ring.full0 + 8 * ((n_req - 1) % NXS), ((n_req - 1) / NXS) & 1, lim) &&
      lane == 0)
    set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
  if (!ok && lane == 0) {
    misc->abort_ = 1;
    set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
  }
  // every issued copy lands before the shared memory is released
  bool drained = true;
  for (uint32_t s = 0; s < (uint32_t)L::NSTG && s < cnt; ++s)
    if (!warp_wait(bar(land0 + s), ((cnt - 1 - s) / L::NSTG) & 1, lim)) drained = false;
  for (uint32_t q = 0; !v_role && q < 2 && q < qi; ++q)
    if (!warp_wait(bar(B_QF + ((qi - 1 - q) & 1)), ((qi - 1 - q) >> 1) & 1, lim)) drained = false;
  if (!drained && lane == 0) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
}

// The converter warps of the E4M3 instantiation (L::NCV for K, as many for V). Tile by tile,
// in copy order, each converts its share of the 128 rows exactly to f16 into the ring stage,
// in the layout the bf16 copies give (row r, 16-byte chunk j of a 64-column half at
// j ^ (r % 8)), frees the staging slot and announces the stage. The first V converter also
// writes the tile's (K, V) page scales beside its V stage (they live as long as the stage);
// the first K converter takes each unit's q to f16 in place after a power-of-two scaling per
// row that brings the row's largest magnitude to [2^14, 2^15) (exact for bf16 values; the
// softmax multiplies by 2^-sh). They wait only on the copies and on the products of earlier
// tiles, never on the next unit.
template <int G>
__device__ __forceinline__ void convert_fp8(const DecodeArgs& a, unsigned char* smem, uint32_t sb, Misc* misc,
                                            const NextRing& ring, const uint16_t* ord, int n_units, int warp,
                                            int lane) {
  using L = TcL<true>;
  auto bar = [&](int i) { return sb + L::SM_BAR + 8 * i; };
  const uint64_t lim = a.wait_limit_ns;
  const bool v_role = warp >= 11 + L::NCV;
  const int ci = (warp - 11) % L::NCV;
  const int land0 = v_role ? B_VT : B_KT, full0 = v_role ? B_VF : B_KF, empty0 = v_role ? B_VE : B_KE,
            sfree0 = v_role ? B_VSE : B_KSE;
  const uint32_t ns = v_role ? L::NSV : L::NSK;
  const unsigned char* stg = smem + (v_role ? L::SM_VS : L::SM_KS);
  unsigned char* ringb = smem + (v_role ? L::SM_V : L::SM_K);
  const int* pages_s = reinterpret_cast<const int*>(smem + L::SM_PH) + 3 * 8;
  float* scales = reinterpret_cast<float*>(smem + L::SM_SC);
  float* qun = reinterpret_cast<float*>(smem + L::SM_QU);
  // half-warp h takes row 2 i + h; lane c of it takes codes 8c .. 8c + 7 (dims 8c .. 8c + 7):
  // the 16 loads of a row read 128 contiguous bytes and the 8 stores of a 64-column half fill
  // one 128-byte row, so neither conflicts on a shared-memory bank
  const int c = lane & 15, hrow = lane >> 4;
  uint32_t cv = 0, qi = 0, k = 0;
  bool ok = true;
  for (int id = blockIdx.x; id < n_units; id = next_item(ring, k++, n_units, a.err_flag)) {
    const Unit u = make_unit(a, id, ord);
    if (u.kind != 0 || !ok) continue;
    if (!v_role && ci == 0) {
      // q: lane pair (2r, 2r + 1) takes row r, 64 columns each (any chunk order: every chunk
      // of the row is read and written back in place)
      const uint32_t qb = qi & 1;
      if (!warp_wait(bar(B_QF + qb), (qi >> 1) & 1, lim)) {
        ok = false;
        continue;
      }
      const int r = lane >> 1;
      unsigned char* qrow = smem + L::SM_Q + qb * QB + (lane & 1) * (QB / 2) + r * 128;
      float mx = 0.0f;
#pragma unroll 2
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + cc * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u))));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      // exponent of mx (0 for zero and subnormals), then sh = 14 - exponent within the
      // normal range of a float scale factor
      const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
      int sh = mx > 0.0f ? 14 - ex : 0;
      sh = sh > 126 ? 126 : (sh < -126 ? -126 : sh);
      const float up = __uint_as_float((uint32_t)(127 + sh) << 23);
#pragma unroll 2
      for (int cc = 0; cc < 8; ++cc) {  // read again: fewer registers held across the two passes
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + cc * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 h =
              __floats2half2_rn(__uint_as_float(w[e] << 16) * up, __uint_as_float(w[e] & 0xffff0000u) * up);
          o[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(qrow + cc * 16) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if ((lane & 1) == 0) qun[qb * NQ + r] = __uint_as_float((uint32_t)(127 - sh) << 23);
      fence_proxy_async_smem();
      __syncwarp();
      if (elect_one()) mbar_arrive(bar(B_QC + qb));
      __syncwarp();
    }
    ++qi;
    for (int j = 0; j < u.n_tiles; ++j, ++cv) {
      const uint32_t slot = cv % L::NSTG, st = cv % ns;
      if (!warp_wait(bar(land0 + slot), (cv / L::NSTG) & 1, lim)) {
        ok = false;
        break;
      }
      float ksc = 1.0f, vsc = 1.0f;
      const bool scaler = v_role && ci == 0 && lane < 8;
      if (scaler) {  // read while the rows are converted
        const size_t si = (size_t)pages_s[slot * 8 + lane] * a.n_kv_heads + u.hk;
        ksc = __ldg(a.k_scale + si);
        vsc = __ldg(a.v_scale + si);
      }
      if (cv >= ns && !warp_wait(bar(empty0 + st), ((cv / ns) - 1) & 1, lim)) {
        ok = false;
        break;
      }
      const unsigned char* s_lane = stg + slot * L::STG + hrow * TD + c * 8;
      unsigned char* d_lane = ringb + st * KVT + (c >> 3) * KVH + hrow * 128;
      // this warp's row pairs [i_lo, i_hi), eight at a time with all eight loads issued first
      // (a load, its conversions and its store in sequence leave the warp waiting on each load)
      constexpr int PER = (TK / 2 + L::NCV - 1) / L::NCV;
      const int i_lo = ci * PER, i_hi = min(TK / 2, i_lo + PER);
      for (int i0 = i_lo; i0 < i_hi; i0 += 8) {
        uint2 w[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (i0 + q < i_hi) w[q] = *reinterpret_cast<const uint2*>(s_lane + (i0 + q) * 2 * TD);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (i0 + q < i_hi) {
            const int i = i0 + q, r = 2 * i + hrow;  // key row
            const uint4 o = make_uint4(e4m3x2_to_f16x2(w[q].x), e4m3x2_to_f16x2(w[q].x >> 16),
                                       e4m3x2_to_f16x2(w[q].y), e4m3x2_to_f16x2(w[q].y >> 16));
            *reinterpret_cast<uint4*>(d_lane + i * 2 * 128 + (((c & 7) ^ (r & 7)) << 4)) = o;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (elect_one()) mbar_arrive(bar(sfree0 + slot));  // this warp has read its rows of the slot
      if (scaler) {
        scales[(st * 8 + lane) * 2] = ksc;
        scales[(st * 8 + lane) * 2 + 1] = vsc;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (elect_one()) mbar_arrive(bar(full0 + st));
      __syncwarp();
    }
  }
  if (!ok && lane == 0) {
    misc->abort_ = 1;
    set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
  }
}

// UNIFIED: FlashDecoding++'s asynchronised softmax with a unified maximum value
// ("【FlashAttention-V4，非官方】FlashDecoding++", sections 1 and 3). Every head's logits are
// exponentiated against the preset phi, so a tile needs no maximum at all: one OR over the
// threads tells whether any logit lies above phi + 60 (natural-log units), or, on a unit's
// first tile, whether a head lies wholly below phi - 60. Only then is the tile's maximum
// taken, the reference moved as in the CUDA-core kernel and the event counted.
//
// CASCADE: the launch follows the shared-prefix kernel of a cascade (a.pre_o is set) and
// each final row merges the prefix's chunk states into its own.
//
// FP8: the pools hold E4M3 codes with per-(page, KV head) scales; the producers bring a tile of
// codes into a staging ring and convert it (exactly) to f16 in the K or V ring, q is taken to
// f16 after a per-row power-of-two scaling, and both products take f16 operands.
template <int G, bool UNIFIED, bool CASCADE, bool FP8>
__global__ void __launch_bounds__(TcL<FP8>::THREADS, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, const DecodeArgs a, int n_units) {
  using L = TcL<FP8>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  Misc* misc = reinterpret_cast<Misc*>(smem + L::SM_MISC);
  auto bar = [&](int i) { return sb + L::SM_BAR + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = a.wait_limit_ns;
  // one split per sequence: hand out the longest sequences' units first
  const bool lpt = a.num_splits == 1 && a.batch > 1 && a.batch <= LPT_MAX;
  int* hist = reinterpret_cast<int*>(smem + L::SM_HIST);
  uint16_t* ord_s = reinterpret_cast<uint16_t*>(smem + L::SM_ORD);
  const int my_bucket = lpt && threadIdx.x < a.batch ? lpt_bucket(a, threadIdx.x) : 0;
  // Without the longest-first order a CTA's first unit is its own index, so the producers
  // request that unit's first 32 table entries now, beside the length reads: its first
  // copies then wait for one round trip to memory, not two. Entries past the split's pages
  // are read but never used; all lie inside the table.
  int ent_first = 0;
  if (!FP8 && !lpt && (warp == 0 || warp == 2)) {
    const int split0 = (int)blockIdx.x % a.num_splits;
    const int b0 = (int)blockIdx.x / a.num_splits / a.n_kv_heads;
    const int idx = split0 * a.pages_per_split + lane;
    if (b0 < a.batch && lane < a.pages_per_split && idx < a.max_blocks)
      ent_first = __ldg(a.block_table + (size_t)b0 * a.max_blocks + idx);
  }
  if (lpt && threadIdx.x < LPT_BUCKETS) hist[threadIdx.x] = 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      int cnt = 1;
      // one arrival from each of the four softmax (or epilogue) warps
      if ((i >= B_SE && i < B_SE + 2) || (i >= B_PF && i < B_PF + 2) || (i >= B_OF && i < B_OF + 2) ||
          (i >= B_STF && i < B_STF + 2) || (i >= B_STE && i < B_STE + 2) || (i >= B_RED && i < B_RED + NRED))
        cnt = 4;
      if (i >= B_NE && i < B_NE + NXS) cnt = L::NWARP;
      // E4M3 pools: a ring stage is announced, and a staging tile freed, by each converter warp
      if (FP8 && ((i >= B_KF && i < B_KF + 3) || (i >= B_VF && i < B_VF + 3) || (i >= B_KSE && i < B_KSE + 3) ||
                  (i >= B_VSE && i < B_VSE + 3)))
        cnt = L::NCV;
      mbar_init(bar(i), cnt);
    }
    misc->abort_ = 0;
    for (int i = 0; i < NBADM; ++i) misc->bad_item[i] = -1;
    fence_mbar_init();
  }
  // P^T rows past the group are never written: keep them zero.
  for (int i = threadIdx.x; i < 2 * PB / 16; i += L::THREADS)
    reinterpret_cast<uint4*>(smem + L::SM_P)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const NextRing ring{smem_u32(&misc->next[0]), bar(B_NF), bar(B_NE)};
  if (lpt) {
    // Stable counting sort of the sequences by tiles, most first. Every CTA must arrive at
    // the same order (a unit id means the same sequence in all of them), so the counts are
    // taken with atomics but the places are given by one warp in sequence order.
    uint8_t* bk = smem + L::SM_BK;
    for (int b = threadIdx.x; b < a.batch; b += L::THREADS) {
      const int key = b == threadIdx.x ? my_bucket : lpt_bucket(a, b);
      bk[b] = (uint8_t)key;
      atomicAdd(&hist[key], 1);
    }
    __syncthreads();
    if (warp == 0) {
      {  // exclusive prefix sum of the 64 counts, two per lane
        const int h0 = hist[2 * lane], h1 = hist[2 * lane + 1];
        int incl = h0 + h1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        hist[2 * lane] = incl - h0 - h1;
        hist[2 * lane + 1] = incl - h1;
      }
      __syncwarp();
      for (int b0 = 0; b0 < a.batch; b0 += 32) {
        const int b = b0 + lane;
        const bool v = b < a.batch;
        const int key = v ? bk[b] : LPT_BUCKETS + lane;  // lanes past the batch match nobody
        const unsigned same = __match_any_sync(0xffffffffu, key);
        if (v) ord_s[hist[key] + __popc(same & ((1u << lane) - 1u))] = (uint16_t)b;
        __syncwarp();
        if (v && lane == 31 - __clz(same)) hist[key] += __popc(same);  // the group's last lane
        __syncwarp();
      }
    }
    __syncthreads();
  }
  const uint16_t* ord = lpt ? ord_s : nullptr;
  // The split merge, launched next on the same stream, may take its place on the SMs once
  // every CTA of this grid has started (or was taken over); it waits for this grid before
  // it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if constexpr (FP8) {
    if (warp == 0 || warp == 2) produce_fp8<G>(a, mq, mk, mv, smem, sb, misc, ring, ord, n_units, warp, lane);
  }
  if (!FP8 && (warp == 0 || warp == 2)) {
    // ------------------------------------------------------------------ TMA producers
    // Warp 0: each unit's Q (double-buffered, so the next unit's Q arrives while this one
    // runs) and K tiles; warp 2: V tiles. Each waits only on its own ring.
    const bool v_role = warp == 2;
    if (elect_one()) {
      tma_prefetch_desc(v_role ? &mv : &mk);
      if (!v_role) tma_prefetch_desc(&mq);
    }
    __syncwarp();
    uint32_t cnt = 0, qi = 0, k = 0, n_req = 0;
    bool ok = true;
    for (int id = blockIdx.x; ok && id < n_units; id = next_item(ring, k++, n_units, a.err_flag)) {
      const Unit u = make_unit(a, id, ord);
      if (u.kind == 0 && !v_role) {
        // Q of the group (rows past the group read other heads' q, or 0 past the last head)
        const uint32_t qb = qi & 1;
        if (qi >= 2 && !warp_wait(bar(B_QE + qb), ((qi >> 1) - 1) & 1, lim)) ok = false;
        if (ok && elect_one()) {
          mbar_arrive_expect_tx(bar(B_QF + qb), QB);
          tma_load_3d(sb + L::SM_Q + qb * QB, &mq, 0, u.hk * G, u.b, bar(B_QF + qb));
          tma_load_3d(sb + L::SM_Q + qb * QB + QB / 2, &mq, 64, u.hk * G, u.b, bar(B_QF + qb));
        }
        __syncwarp();
      }
      if (u.kind == 0) ++qi;
      if (!v_role && ok) {
        // ask for the next unit as soon as this one is known, so that the answer is in by
        // the time this unit's copies are issued (units can be one tile long)
        const uint32_t s = k % NXS, uu = k / NXS;
        if (uu > 0 && !warp_wait(ring.empty0 + 8 * s, (uu - 1) & 1, lim)) ok = false;
        if (ok) {
          if (elect_one()) request_next_cta(ring.slot0 + 16 * s, ring.full0 + 8 * s);
          __syncwarp();
          ++n_req;
        }
      }
      // The unit's table entries, 32 pages (four tiles) per warp-wide load: lane l holds
      // page 32 c + l of the split; a tile's page pp comes from lane (8 j + pp) % 32.
      const int32_t* trow = a.block_table + (size_t)u.b * a.max_blocks + u.first;
      int ent = 0;
      for (int j = 0; ok && j < u.n_tiles; ++j, ++cnt) {
        if ((j & 3) == 0)
          ent = (32 * (j >> 2) + lane < u.n_pages)
                    ? ((k == 0 && j == 0 && !lpt) ? ent_first : __ldg(trow + 32 * (j >> 2) + lane))
                    : 0;
        const uint32_t s = cnt % L::NSK, use = cnt / L::NSK;
        const uint32_t full = bar((v_role ? B_VF : B_KF) + s);
        if (use > 0 && !warp_wait(bar((v_role ? B_VE : B_KE) + s), (use - 1) & 1, lim)) {
          ok = false;
          break;
        }
        if (__any_sync(0xffffffffu, misc->abort_ != 0)) {
          ok = false;
          break;
        }
        // lane pp < 8 takes the entry of the tile's page pp (slots past the split reload a
        // page of the unit: finite data, masked)
        const int pages = min(8, u.n_pages - 8 * j);
        // (both shuffles are taken by the whole warp; a shuffle under a lane-dependent
        // condition with a full mask is undefined)
        const int own = __shfl_sync(0xffffffffu, ent, (8 * j + (lane & 7)) & 31);
        const int tile_first = __shfl_sync(0xffffffffu, ent, (8 * j) & 31);
        int phys = lane < pages ? own : tile_first;
        bool bad = false;
        if (lane < 8) {
          bad = phys < 0 || phys >= a.num_pages;
          if (bad) phys = 0;
        }
        const bool any_bad = __any_sync(0xffffffffu, bad);
        if (any_bad && lane == 0) {
          misc->bad_item[k % NBADM] = id;  // written before the arrival that publishes the tile
          set_err(a.err_flag, PKV_DEVERR_BAD_PAGE);
        }
        const uint32_t dst = sb + (v_role ? L::SM_V : L::SM_K) + s * KVT;
        const CUtensorMap* map = v_role ? &mv : &mk;
        const bool stall = !v_role && a.stall_page >= 8 * j && a.stall_page < 8 * j + 8;
        __syncwarp();
        if (lane == 0 && !stall) mbar_arrive_expect_tx(full, KVT);
        __syncwarp();
        if (lane < 8 && !stall) {
          const int row = (phys * a.n_kv_heads + u.hk) * 16;
          tma_load_2d(dst + lane * 2048, map, 0, row, full);
          tma_load_2d(dst + KVH + lane * 2048, map, 64, row, full);
        }
        __syncwarp();
      }
    }
    if (!v_role && n_req > k && !warp_wait(ring.full0 + 8 * ((n_req - 1) % NXS), ((n_req - 1) / NXS) & 1, lim) &&
        lane == 0)
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    if (!ok && lane == 0) {
      misc->abort_ = 1;
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
    // every issued copy lands before the shared memory is released (the consumers normally
    // waited for them already)
    bool drained = true;
    const uint32_t ns = v_role ? L::NSV : L::NSK;
    for (uint32_t s = 0; s < ns && s < cnt; ++s)
      if (!warp_wait(bar((v_role ? B_VF : B_KF) + s), ((cnt - 1 - s) / ns) & 1, lim)) drained = false;
    for (uint32_t q = 0; !v_role && q < 2 && q < qi; ++q)
      if (!warp_wait(bar(B_QF + ((qi - 1 - q) & 1)), ((qi - 1 - q) >> 1) & 1, lim)) drained = false;
    if (!drained && lane == 0) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
  } else if (warp == 0 || warp == 2) {
    // (E4M3 pools: the producers ran above)
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // E4M3 pools: both products take f16 operands (format 0 in the A and B fields)
    constexpr uint32_t kF16 = FP8 ? ((1u << 7) | (1u << 10)) : 0u;
    const uint32_t idS = idesc_bf16_f32(TK, NQ, false, false) & ~kF16;
    const uint32_t idPV = idesc_bf16_f32(TD, NQ, true, false) & ~kF16;
    const uint64_t dk0 = smem_desc(sb + L::SM_K, 16, 1024, kSwizzle128B);
    const uint64_t dq0 = smem_desc(sb + L::SM_Q, 16, 1024, kSwizzle128B);
    const uint64_t dv0 = smem_desc(sb + L::SM_V, KVH, 1024, kSwizzle128B);
    const uint64_t dp0 = smem_desc(sb + L::SM_P, 16, 1024, kSwizzle128B);
    uint32_t k_cnt = 0, v_cnt = 0, g = 0, qi = 0, k = 0;
    bool ok = true;
    // PV of global step gp (tile jp of unit qi): O^T[qi & 1] (+)= V^T P^T
    auto issue_pv = [&](uint32_t gp, int jp) -> bool {
      if (!warp_wait(bar(B_PF + (gp & 1)), (gp >> 1) & 1, lim)) return false;
      const uint32_t vg = v_cnt + jp;
      if (!warp_wait(bar(B_VF + vg % L::NSV), (vg / L::NSV) & 1, lim)) return false;
      // O^T[qi & 1] was last read by the epilogue of unit qi - 2
      if (jp == 0 && qi >= 2 && !warp_wait(bar(B_OF + (qi & 1)), ((qi >> 1) - 1) & 1, lim)) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dv = dv0 + (uint64_t)((vg % L::NSV) * KVT >> 4);
        const uint64_t dp = dp0 + (uint64_t)(((gp & 1) * PB) >> 4);
#pragma unroll
        for (int kk = 0; kk < TK / 16; ++kk)
          mma_bf16_ss(tmem + COL_O + (qi & 1) * NQ, dv + (uint64_t)((kk * 2048) >> 4),
                      dp + (uint64_t)(((kk / 4) * (PB / 2) + (kk % 4) * 32) >> 4), idPV,
                      (jp > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(B_OD));
        mma_commit(bar(B_VE + vg % L::NSV));
        mma_commit(bar(B_PE + (gp & 1)));
      }
      __syncwarp();
      return true;
    };
    for (int id = blockIdx.x; ok && id < n_units; id = next_item(ring, k++, n_units, a.err_flag)) {
      const Unit u = make_unit(a, id, ord);
      if (u.kind != 0) continue;
      const uint32_t qb = qi & 1;
      if (!warp_wait(bar((FP8 ? B_QC : B_QF) + qb), (qi >> 1) & 1, lim)) {
        ok = false;
        break;
      }
      const uint32_t g0 = g;
      for (int j = 0; j < u.n_tiles; ++j, ++g) {
        const uint32_t kg = k_cnt + j;
        if (!warp_wait(bar(B_KF + kg % L::NSK), (kg / L::NSK) & 1, lim)) { ok = false; break; }
        if (g >= 2 && !warp_wait(bar(B_SE + (g & 1)), ((g >> 1) - 1) & 1, lim)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dk = dk0 + (uint64_t)((kg % L::NSK) * KVT >> 4);
          const uint64_t dq = dq0 + (uint64_t)((qb * QB) >> 4);
#pragma unroll
          for (int kk = 0; kk < TD / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk / 4) * KVH + (kk % 4) * 32) >> 4);
            const uint64_t offq = (uint64_t)(((kk / 4) * (QB / 2) + (kk % 4) * 32) >> 4);
            mma_bf16_ss(tmem + COL_S + (g & 1) * NQ, dk + off, dq + offq, idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SF + (g & 1)));
          mma_commit(bar(B_KE + kg % L::NSK));
          if (j == u.n_tiles - 1) mma_commit(bar(B_QE + qb));  // the unit's last product that reads Q
        }
        __syncwarp();
        if (j >= 1 && !issue_pv(g - 1, j - 1)) { ok = false; break; }
      }
      if (!ok) break;
      if (!issue_pv(g0 + u.n_tiles - 1, u.n_tiles - 1)) { ok = false; break; }
      if (elect_one()) mma_commit(bar(B_UD + qb));
      __syncwarp();
      k_cnt += u.n_tiles;
      v_cnt += u.n_tiles;
      ++qi;
    }
    if (!ok && lane == 0) {
      misc->abort_ = 1;
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
    // every issued product finishes before TMEM is freed
    if (elect_one()) mma_commit(bar(B_DR));
    __syncwarp();
    if (!warp_wait(bar(B_DR), 0, lim) && lane == 0) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
  } else if (warp < 7) {
    // ------------------------------------------------------------------ softmax
    const int wq = warp & 3;           // TMEM lane quarter of this warp
    const int t = wq * 32 + lane;      // key of a tile
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    const float c = a.scale * kL2e;
    float* red = reinterpret_cast<float*>(smem + L::SM_RED);
    float* stats = reinterpret_cast<float*>(smem + L::SM_ST);
    uint32_t g = 0, v_cnt = 0, qi = 0, k = 0, n_fb = 0;
    bool ok = true;
    for (int id = blockIdx.x; id < n_units; id = next_item(ring, k++, n_units, a.err_flag)) {
      const Unit u = make_unit(a, id, ord);
      if (u.kind != 0 || !ok) continue;  // the epilogue warps write the rows of the other units
      const uint32_t qb = qi & 1;
      float M[G], lp[G], cq[G];  // cq: the logit scale of each head (E4M3 pools: with its q's 2^-sh)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        M[h] = UNIFIED ? a.phi * kL2e : -INFINITY;
        lp[h] = 0.0f;
        cq[h] = c;
      }
      if constexpr (FP8) {
        if (!warp_wait(bar(B_QC + qb), (qi >> 1) & 1, lim)) {
          ok = false;
          continue;
        }
        const float* qun = reinterpret_cast<const float*>(smem + L::SM_QU) + qb * NQ;
#pragma unroll
        for (int h = 0; h < G; ++h) cq[h] = c * qun[h];
      }
      for (int j = 0; j < u.n_tiles; ++j, ++g) {
        const uint32_t bsel = g & 1;
        if (!warp_wait(bar(B_SF + bsel), (g >> 1) & 1, lim)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[NQ];
        tmem_ld16(tmem + lane_addr + COL_S + bsel * NQ, sr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (elect_one()) mbar_arrive(bar(B_SE + bsel));
        __syncwarp();
        const int valid = tile_valid(u, j);
        float ks = 1.0f, vsc = 1.0f;  // E4M3 pools: the K and V scales of key t's page
        if constexpr (FP8) {
          // the V stage's conversion carries the tile's page scales
          const uint32_t vg = v_cnt + j;
          if (!warp_wait(bar(B_VF + vg % L::NSV), (vg / L::NSV) & 1, lim)) { ok = false; break; }
          const float* sc = reinterpret_cast<const float*>(smem + L::SM_SC) + ((vg % L::NSV) * 8 + (t >> 4)) * 2;
          ks = sc[0];
          vsc = sc[1];
        }
        float x[G], mt[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          x[h] = t < valid ? __uint_as_float(sr[h]) * (FP8 ? cq[h] * ks : c) : -INFINITY;
          mt[h] = x[h];
        }
        bool need = false, raise = false;  // the same on every thread
        float alpha[G];
        if constexpr (UNIFIED) {
          // bit 31: a logit above its reference + beta; bit h (first tile): some key of head
          // h is not below its reference - beta (masked keys are -inf, never)
          const float beta2 = kUnifiedBetaTc * kL2e;
          uint32_t w = 0;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if (x[h] > M[h] + beta2) w |= 1u << 31;
            if (j == 0 && x[h] >= M[h] - beta2) w |= 1u << h;
          }
          if (!block_or(w, red, bsel, bar(B_RED + bsel), g >> 1, wq, lane, lim)) { ok = false; break; }
          const uint32_t low_heads = j == 0 ? (~w) & ((1u << G) - 1u) : 0u;
          if ((w >> 31) || low_heads) {
            const int sel = 3 + (n_fb & 1);
            if (!block_reduce<G, true>(mt, red, sel, bar(B_RED + sel), n_fb >> 1, wq, lane, lim)) { ok = false; break; }
            ++n_fb;
            int events = 0;
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const bool hi = mt[h] > M[h] + beta2;
              const bool lo = j == 0 && mt[h] < M[h] - beta2;
              alpha[h] = hi ? ex2(M[h] - mt[h]) : 1.0f;  // nothing is accumulated yet when lo
              if (hi) raise = true;
              if (hi || lo) {
                lp[h] *= alpha[h];
                M[h] = mt[h];
                ++events;
              }
            }
            need = raise;
            if (events && t == 0 && a.fallback_count) atomicAdd(a.fallback_count, events);
          }
        } else {
          if (!block_reduce<G, true>(mt, red, bsel, bar(B_RED + bsel), g >> 1, wq, lane, lim)) { ok = false; break; }
#pragma unroll
          for (int h = 0; h < G; ++h) need |= mt[h] > M[h] + kSlack;
          if (need) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float mn = mt[h] > M[h] + kSlack ? mt[h] : M[h];
              alpha[h] = ex2(M[h] - mn);  // 0 while M = -inf
              lp[h] *= alpha[h];
              M[h] = mn;
            }
          }
        }
        if (need && j > 0) {
          // O^T changes only once PV of the previous step is done (this step's S came after
          // the PV two steps back, so that one is the only product pending)
          if (!warp_wait(bar(B_OD), (g - 1) & 1, lim)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[NQ];
          tmem_ld16(tmem + lane_addr + COL_O + qb * NQ, o);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
          tmem_st16(tmem + lane_addr + COL_O + qb * NQ, o);
          tmem_st_wait();
        }
        // P^T for this step, bf16, key t in column t of each head's row (128-byte swizzle)
        if (g >= 2 && !warp_wait(bar(B_PE + bsel), ((g >> 1) - 1) & 1, lim)) { ok = false; break; }
        unsigned char* pbuf = smem + L::SM_P + bsel * PB + (t >> 6) * (PB / 2);
        const int within = t & 63, chunk = within >> 3;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = ex2(x[h] - M[h]);
          lp[h] += p;
          unsigned short* dstp = reinterpret_cast<unsigned short*>(pbuf + (h >> 3) * 1024 + (h & 7) * 128 +
                                                                   ((chunk ^ (h & 7)) << 4) + (within & 7) * 2);
          // E4M3 pools: the weight times its page's V scale, in f16 (the V tile holds the codes)
          *dstp = FP8 ? __half_as_ushort(__float2half_rn(p * vsc)) : __bfloat16_as_ushort(__float2bfloat16_rn(p));
        }
        if (valid < TK) {
          // masked keys enter PV as 0 x V: the V rows past the sequence (not the caller's
          // data, maybe not finite) are zeroed once the tile has landed
          const uint32_t vg = v_cnt + j;
          if (!warp_wait(bar(B_VF + vg % L::NSV), (vg / L::NSV) & 1, lim)) { ok = false; break; }
          if (t >= valid) {
            unsigned char* vrow = smem + L::SM_V + (vg % L::NSV) * KVT + t * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              reinterpret_cast<uint4*>(vrow)[i] = make_uint4(0u, 0u, 0u, 0u);
              reinterpret_cast<uint4*>(vrow + KVH)[i] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (elect_one()) mbar_arrive(bar(B_PF + bsel));
        __syncwarp();
      }
      if (!ok) continue;
      v_cnt += u.n_tiles;
      // the unit's statistics for the epilogue warps: each head's reference max and sum
      if (!block_reduce<G, false>(lp, red, 2, bar(B_RED + 2), qi, wq, lane, lim)) {
        ok = false;
        continue;
      }
      if (qi >= 2 && !warp_wait(bar(B_STE + qb), ((qi >> 1) - 1) & 1, lim)) {
        ok = false;
        continue;
      }
      if (t < G) {
        float mh = M[0], lh = lp[0];
#pragma unroll
        for (int h = 1; h < G; ++h) {
          mh = t == h ? M[h] : mh;
          lh = t == h ? lp[h] : lh;
        }
        stats[(qb * NQ + t) * 2] = mh;
        stats[(qb * NQ + t) * 2 + 1] = lh;
      }
      __syncwarp();
      if (elect_one()) mbar_arrive(bar(B_STF + qb));
      __syncwarp();
      ++qi;
    }
    if (!ok && lane == 0) {
      misc->abort_ = 1;
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp < 11) {
    // ------------------------------------------------------------------ epilogue
    // Thread t holds head dim t of O^T. Per unit: wait for its last PV and its statistics,
    // read O^T (the buffer is then free for unit + 2), write out / lse or the partial state.
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    const float* stats = reinterpret_cast<const float*>(smem + L::SM_ST);
    uint32_t qi = 0, k = 0;
    bool ok = true;
    bool pre_ready = !CASCADE;  // cascade: the prefix kernel's results may be read
    auto wait_prefix = [&]() {
      if (!pre_ready) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        pre_ready = true;
      }
    };
    for (int id = blockIdx.x; id < n_units; id = next_item(ring, k++, n_units, a.err_flag)) {
      const Unit u = make_unit(a, id, ord);
      const size_t row0 = (size_t)u.b * a.n_qo_heads + (size_t)u.hk * G;  // the group's first row
      if (u.kind == 1 || u.kind == 2) {
        const float o = u.kind == 1 ? NAN : 0.0f, l = u.kind == 1 ? NAN : -INFINITY;
        if (u.kind == 1 && t == 0) set_err(a.err_flag, PKV_DEVERR_BAD_LEN);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
        float vals[G], lses[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          vals[h] = o;
          lses[h] = l;
        }
        if (CASCADE && u.kind == 2) {  // no suffix keys: the prefix alone
          wait_prefix();
          cascade_merge_group<G>(a, row0, t, vals, lses);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          out[(row0 + h) * TD + t] = __float2bfloat16_rn(vals[h]);
          if (a.lse && t == h) a.lse[row0 + h] = lses[h];
        }
        continue;
      }
      if (u.kind != 0) continue;
      const uint32_t qb = qi & 1;
      ++qi;
      float o[G], mh[G], lh[G];
      bool good = false;
      if (ok) {
        ok = warp_wait(bar(B_STF + qb), ((qi - 1) >> 1) & 1, lim) && warp_wait(bar(B_UD + qb), ((qi - 1) >> 1) & 1, lim);
        tc_fence_after();
        uint32_t r[NQ];
        tmem_ld16(tmem + lane_addr + COL_O + qb * NQ, r);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < G; ++h) {
          o[h] = __uint_as_float(r[h]);
          mh[h] = stats[(qb * NQ + h) * 2];
          lh[h] = stats[(qb * NQ + h) * 2 + 1];
        }
        tc_fence_before();
        __syncwarp();
        if (elect_one()) {
          mbar_arrive(bar(B_OF + qb));   // O^T[qb] may take unit qi + 1's products
          mbar_arrive(bar(B_STE + qb));  // the statistics buffer may take unit qi + 1's
        }
        __syncwarp();
        good = ok && *reinterpret_cast<volatile int*>(&misc->bad_item[k % NBADM]) != id;
        if (!ok && lane == 0) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
      }
      float vals[G], lses[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        vals[h] = good ? o[h] / lh[h] : NAN;
        lses[h] = good ? (mh[h] + log2f(lh[h])) * kLn2 : NAN;
      }
      if (CASCADE && u.final_write) {
        wait_prefix();
        cascade_merge_group<G>(a, row0, t, vals, lses);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float val = vals[h], lse = lses[h];
        const size_t row = row0 + h;
        if (u.final_write) {
          static_cast<__nv_bfloat16*>(a.out)[row * TD + t] = __float2bfloat16_rn(val);
          if (a.lse && t == h) a.lse[row] = lse;
        } else {
          a.part_o[(row * a.num_splits + u.split) * TD + t] = val;
          if (t == h) a.part_lse[row * a.num_splits + u.split] = lse;
        }
      }
    }
  } else if constexpr (FP8) {
    // ------------------------------------------------------------------ converters (E4M3)
    convert_fp8<G>(a, smem, sb, misc, ring, ord, n_units, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  // cascade: a CTA whose units never read the prefix's states still ends only after the
  // prefix grid, so that this grid never ends before it
  if (CASCADE) asm volatile("griddepcontrol.wait;" ::: "memory");
}

bool encode_map(CUtensorMap* m, CUtensorMapDataType type, CUtensorMapSwizzle swz, const void* ptr, int rank,
                const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, type, rank, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G, bool UNIFIED, bool CASCADE, bool FP8>
int launch_tc(const DecodeArgs& a, cudaStream_t stream) {
  using L = TcL<FP8>;
  CUtensorMap mq, mk, mv;
  {
    // q [B][Hq][128] as (128, Hq, B): a box is 64 columns of 16 heads of one sequence
    cuuint64_t dims[3] = {(cuuint64_t)TD, (cuuint64_t)a.n_qo_heads, (cuuint64_t)a.batch};
    cuuint64_t strides[2] = {(cuuint64_t)TD * 2, (cuuint64_t)a.n_qo_heads * TD * 2};
    cuuint32_t box[3] = {64, NQ, 1};
    if (!encode_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, a.q, 3, dims, strides, box))
      return check_launch(cudaErrorInvalidValue);
  }
  {
    // pools [pages][Hkv][16][128] as rows of 128: bf16, a box is one (page, KV head) block of
    // 16 rows x 64 columns in the 128-byte swizzle; E4M3, a box is the block's 16 rows of 128
    // codes, unswizzled (the producer converts them into the swizzled f16 layout)
    const cuuint64_t rows = (cuuint64_t)a.num_pages * a.n_kv_heads * 16;
    cuuint64_t dims[2] = {(cuuint64_t)TD, rows};
    cuuint64_t strides[1] = {(cuuint64_t)TD * (FP8 ? 1 : 2)};
    cuuint32_t box[2] = {FP8 ? (cuuint32_t)TD : 64u, 16};
    const CUtensorMapDataType type = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle swz = FP8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!encode_map(&mk, type, swz, a.k_pages, 2, dims, strides, box) ||
        !encode_map(&mv, type, swz, a.v_pages, 2, dims, strides, box))
      return check_launch(cudaErrorInvalidValue);
  }
  static FuncConfigured configured;
  if (!configured.ensure(reinterpret_cast<const void*>(decode_tc_kernel<G, UNIFIED, CASCADE, FP8>), L::SMEM))
    return PKV_ERR_LAUNCH;
  const long n_units = (long)a.num_splits * a.n_kv_heads * a.batch;
  if (n_units <= 0) return PKV_OK;
  if (n_units > 0x7fffffffL) return PKV_ERR_UNSUPPORTED;
  if (!CASCADE) {
    decode_tc_kernel<G, UNIFIED, CASCADE, FP8><<<(unsigned)n_units, L::THREADS, L::SMEM, stream>>>(mq, mk, mv, a,
                                                                                             (int)n_units);
    return check_launch(cudaGetLastError());
  }
  // cascade: may start while the prefix kernel before it finishes (it waits for that grid
  // before reading the prefix's partial states)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)n_units, 1, 1);
  cfg.blockDim = dim3(L::THREADS, 1, 1);
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return check_launch(cudaLaunchKernelEx(&cfg, decode_tc_kernel<G, UNIFIED, CASCADE, FP8>, mq, mk, mv, a, (int)n_units));
}

}  // namespace

bool decode_tc_supported(const DecodeArgs& a) {
  if (a.n_kv_heads <= 0 || a.n_qo_heads % a.n_kv_heads) return false;
  const int G = a.n_qo_heads / a.n_kv_heads;
  if (a.dtype != PKV_BF16 || a.head_dim != TD || a.page_size != 16) return false;
  // E4M3 pools: groups of 4 and 8 (exact softmax, not a cascade's suffix). With 1 or 2 query
  // heads per KV head the CUDA-core kernel, which reads the codes straight from its ring, is
  // faster: there the conversion to f16 and the extra shared-memory traffic it costs are not
  // paid back by the products (measured on the Llama-7B batch: 76 us against 114; with 4 heads
  // per KV head the two are equal, with 8 the tensor cores are 3x faster).
  if (a.fp8) return (G == 4 || G == 8) && !a.unified && !a.pre_o;
  return G == 4 || G == 8;
}

int launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  const int G = a.n_qo_heads / a.n_kv_heads;
  if (a.fp8) {
    if (a.unified || a.pre_o) return PKV_ERR_UNSUPPORTED;
    if (G == 4) return launch_tc<4, false, false, true>(a, stream);
    if (G == 8) return launch_tc<8, false, false, true>(a, stream);
    return PKV_ERR_UNSUPPORTED;
  }
  if (a.pre_o) {  // the suffix of a cascade (exact softmax only)
    if (a.unified) return PKV_ERR_UNSUPPORTED;
    if (G == 4) return launch_tc<4, false, true, false>(a, stream);
    if (G == 8) return launch_tc<8, false, true, false>(a, stream);
    return PKV_ERR_UNSUPPORTED;
  }
  if (G == 4) return a.unified ? launch_tc<4, true, false, false>(a, stream) : launch_tc<4, false, false, false>(a, stream);
  if (G == 8) return a.unified ? launch_tc<8, true, false, false>(a, stream) : launch_tc<8, false, false, false>(a, stream);
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
