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
};

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

// The softmax warpgroup of one query tile: S -> P for every key tile, then the epilogue.
__device__ __forceinline__ void softmax_tile(const PrefillArgs& a, Misc* misc, uint32_t bar_sf,
                                             uint32_t bar_pf, uint32_t bar_od, uint32_t col_s,
                                             uint32_t col_o, int n_tiles, int q0, int b, int h,
                                             int warp, int lane) {
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // row in the tile = TMEM lane
  const uint32_t lane_addr = ((uint32_t)(quarter * 32) << 16);
  const uint32_t tS = misc->tmem_base + lane_addr + col_s;
  const uint32_t tO = misc->tmem_base + lane_addr + col_o;
  const float c = a.scale * kLog2eF;  // logits in log2 units: s * c
  float ms = -INFINITY;               // reference max, log2 units
  float l = 0.0f;
  bool ok = true;
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
    if (jj == n_tiles - 1) {  // diagonal tile: key column c is visible to row r iff c <= r
#pragma unroll
      for (int i = 0; i < 128; ++i) x[i] = (i > r) ? -INFINITY : x[i];
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
  const int t = q0 + r;
  const bool store = t < a.seq_len;  // rows past a ragged end are computed but not stored
  const int H = a.n_qo_heads;
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + (((size_t)b * a.seq_len + t) * H + h) * HD;
  const float inv = ok ? 1.0f / l : NAN;
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
  if (store && a.lse) a.lse[((size_t)b * H + h) * a.seq_len + t] = ok ? (ms + log2f(l)) * kLn2F : NAN;
}

__global__ void __launch_bounds__(THREADS, 1)
prefill_causal_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv, const PrefillArgs a) {
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
  const int n_qt = (a.seq_len + BM - 1) / BM;
  const int n_pairs = (n_qt + 1) / 2;
  // Longest-first order: the pairs nearest the end of the sequence have the most key tiles.
  const int id = blockIdx.x;
  const int pr = n_pairs - 1 - id / (H * a.batch);
  const int rem = id % (H * a.batch);
  const int h = rem % H;
  const int b = rem / H;
  const int hk = h / G;
  const int qtA = 2 * pr;
  const bool has_b = (qtA + 1) < n_qt;
  const int lastA = qtA;                       // A's diagonal key tile
  const int n_kv = has_b ? qtA + 2 : qtA + 1;  // key tiles the CTA walks

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == BAR_PF || i == BAR_PF + 1) ? 128 : 1);
    misc->abort_ = 0;
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
        tma_load_4d(sb + SM_Q + t * TILE, &mq, 0, h, (qtA + t) * BM, b, bar(BAR_Q));
        tma_load_4d(sb + SM_Q + t * TILE + SUB, &mq, 64, h, (qtA + t) * BM, b, bar(BAR_Q));
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
        const int k0 = j * BN;
        tma_load_4d(sb + SM_K + s * TILE, &mk, 0, hk, k0, b, bar(BAR_KVF + s));
        tma_load_4d(sb + SM_K + s * TILE + SUB, &mk, 64, hk, k0, b, bar(BAR_KVF + s));
        tma_load_4d(sb + SM_V + s * TILE, &mv, 0, hk, k0, b, bar(BAR_KVF + s));
        tma_load_4d(sb + SM_V + s * TILE + SUB, &mv, 64, hk, k0, b, bar(BAR_KVF + s));
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
    softmax_tile(a, misc, bar(BAR_SF + 0), bar(BAR_PF + 0), bar(BAR_OD + 0), COL_S, COL_O,
                 lastA + 1, qtA * BM, b, h, warp, lane);
  } else if (has_b) {
    softmax_tile(a, misc, bar(BAR_SF + 1), bar(BAR_PF + 1), bar(BAR_OD + 1), COL_S + BN,
                 COL_O + HD, n_kv, (qtA + 1) * BM, b, h, warp, lane);
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

// [B, T, H, D] bf16 viewed as a 4-D tensor (D, H, T, B); a box is 64 columns x 128 rows of one head.
bool make_btHd_map(CUtensorMap* m, const void* ptr, int B, int T, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)H * HD * 2, (cuuint64_t)T * H * HD * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.head_dim != HD) return PKV_ERR_UNSUPPORTED;
  const long n_qt = (a.seq_len + BM - 1) / BM;
  const long grid = (n_qt + 1) / 2 * a.n_qo_heads * a.batch;
  if (grid > 0x7fffffffL) return PKV_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!make_btHd_map(&mq, a.q, a.batch, a.seq_len, a.n_qo_heads) ||
      !make_btHd_map(&mk, a.k, a.batch, a.seq_len, a.n_kv_heads) ||
      !make_btHd_map(&mv, a.v, a.batch, a.seq_len, a.n_kv_heads))
    return PKV_ERR_LAUNCH;
  static int configured_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 32 && !(configured_mask & (1 << dev))) {
    if (check_launch(cudaFuncSetAttribute(prefill_causal_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)) != PKV_OK)
      return PKV_ERR_LAUNCH;
    configured_mask |= (1 << dev);
  }
  prefill_causal_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, a);
  return check_launch(cudaGetLastError());
}

}  // namespace pkv
