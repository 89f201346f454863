// Causal prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Tiled FlashAttention ("快速注意力内核与算子融合", Q&A on FlashAttention): for
// one (batch, head, 128-row query tile) a CTA walks the 128-key K/V tiles up
// to the diagonal. It computes S = Q K^T into tensor memory, updates the
// running row max and sum, writes P = exp(S - m) back into tensor memory as
// bf16, and accumulates O += P V into tensor memory. The T x T score matrix
// never leaves the chip. The causal mask is applied by predication on the
// diagonal tile only.
//
// Warp roles (192 threads):
//   warp 0    TMA producer (Q once, K/V tiles into a 2-stage ring); owns TMEM
//   warp 1    MMA issuer (one elected thread)
//   warps 2-5 softmax: one thread per query row. Warp w reads TMEM lanes
//             32*(w%4) .. 32*(w%4)+31, so the four warps cover all 128 rows.
// TMEM columns: S buffer 0 [0,128), S buffer 1 [128,256), O [256,384).
// P_j overwrites the first 64 columns of its own S buffer (packed bf16 pairs).
// The PV product reads A = P from TMEM and B = V from shared memory.
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
constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + TILE;
constexpr int SM_V = SM_K + NST * TILE;
constexpr int SM_BAR = SM_V + NST * TILE;
// barriers: q_full, kv_full[2], kv_empty[2], s_full[2], p_full, o_done, mma drain
constexpr int BAR_Q = 0, BAR_KVF = 1, BAR_KVE = 3, BAR_SF = 5, BAR_PF = 7, BAR_OD = 8, BAR_DRAIN = 9,
              NBAR = 10;
constexpr int SM_MISC = SM_BAR + NBAR * 8;
constexpr int SMEM_BYTES = SM_MISC + 64 + 1024;  // + slack to align the base to 1024
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int COL_S0 = 0, COL_O = 256;
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

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
  // Longest-first order: the query tiles nearest the end of the sequence have the most key tiles.
  const int id = blockIdx.x;
  const int qt = n_qt - 1 - id / (H * a.batch);
  const int rem = id % (H * a.batch);
  const int h = rem % H;
  const int b = rem / H;
  const int hk = h / G;
  const int q0 = qt * BM;
  const int n_kv = qt + 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), i == BAR_PF ? 128 : 1);
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
      mbar_arrive_expect_tx(bar(BAR_Q), TILE);
      tma_load_4d(sb + SM_Q, &mq, 0, h, q0, b, bar(BAR_Q));
      tma_load_4d(sb + SM_Q + SUB, &mq, 64, h, q0, b, bar(BAR_Q));
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
        if (!mbar_wait(bar(BAR_KVF + s), ((issued - 1 - s) / NST) & 1)) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
      const uint32_t idPV = idesc_bf16_f32(BM, HD, false, true);
      auto issue_s = [&](int j) {
        const int s = j % NST;
        const uint32_t kb = sb + SM_K + s * TILE;
        const uint32_t d = tmem + COL_S0 + (j & 1) * BN;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k / 4) * SUB + (k % 4) * 32;
          mma_bf16_ss(d, smem_desc(sb + SM_Q + off, 16, 1024, kSwizzle128B),
                      smem_desc(kb + off, 16, 1024, kSwizzle128B), idS, k > 0);
        }
        mma_commit(bar(BAR_SF + (j & 1)));
      };
      bool ok = mbar_wait(bar(BAR_Q), 0) && mbar_wait(bar(BAR_KVF + 0), 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int s = (j + 1) % NST;
          if (!mbar_wait(bar(BAR_KVF + s), ((j + 1) / NST) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(bar(BAR_PF), j & 1)) { ok = false; break; }
        tc_fence_after();
        const int s = j % NST;
        const uint32_t vb = sb + SM_V + s * TILE;
        const uint32_t pcol = tmem + COL_S0 + (j & 1) * BN;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ts(tmem + COL_O, pcol + k * 8, smem_desc(vb + k * 2048, 16384, 1024, kSwizzle128B),
                      idPV, (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(BAR_OD));
        mma_commit(bar(BAR_KVE + s));
      }
      if (!ok) fail(misc, a.err_flag);
      // Every issued product must finish before TMEM is freed.
      mma_commit(bar(BAR_DRAIN));
      if (!mbar_wait(bar(BAR_DRAIN), 0)) set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row in the tile = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const float c = a.scale * kLog2eF;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(bar(BAR_SF + (j & 1)), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t scol = lane_addr + COL_S0 + (j & 1) * BN;
      uint32_t sr[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(scol + q * 32, sr[q]);
      tmem_ld_wait();
      float x[128];
      const bool diag = (j == qt);
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int col = q * 32 + i;
          const float v = __uint_as_float(sr[q][i]) * c;
          x[col] = (diag && col > r) ? -INFINITY : v;
        }
      float mt = x[0];
#pragma unroll
      for (int i = 1; i < 128; ++i) mt = fmaxf(mt, x[i]);
      const float m_new = fmaxf(m, mt);
      const float alpha = ex2(m - m_new);  // 0 on the first tile (m = -inf)
      float rs = 0.0f;
      uint32_t pk[2][32];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float p0 = ex2(x[2 * i] - m_new);
        const float p1 = ex2(x[2 * i + 1] - m_new);
        rs += p0 + p1;
        pk[i / 32][i % 32] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      if (j > 0) {
        // O holds the sum up to tile j-1 once PV_{j-1} is done; rescale it to the new max.
        if (!warp_wait(bar(BAR_OD), (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, m_new > m)) {  // warp-uniform; alpha is 1 where the max held
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(lane_addr + COL_O + q * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_addr + COL_O + q * 32, o);
          }
        }
      }
      m = m_new;
      tmem_st32(scol, pk[0]);
      tmem_st32(scol + 32, pk[1]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(BAR_PF));
    }
    // ------------------------------------------------------------------ epilogue
    ok = __all_sync(0xffffffffu, ok);
    if (ok && !warp_wait(bar(BAR_OD), (n_kv - 1) & 1)) ok = false;
    tc_fence_after();
    const int t = q0 + r;
    if (!ok && lane == 0) fail(misc, a.err_flag);
    const bool store = t < a.seq_len;  // rows past a ragged end are computed but not stored
    const size_t row = ((size_t)b * a.seq_len + t) * H + h;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + row * HD;
    const float inv = ok ? 1.0f / l : NAN;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o[32];
      tmem_ld32(lane_addr + COL_O + q * 32, o);  // all lanes, uniformly
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
    if (store && a.lse) a.lse[((size_t)b * H + h) * a.seq_len + t] = ok ? (m + log2f(l)) * kLn2F : NAN;
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
  const long grid = n_qt * a.n_qo_heads * a.batch;
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
    if (cudaFuncSetAttribute(prefill_causal_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return PKV_ERR_LAUNCH;
    configured_mask |= (1 << dev);
  }
  prefill_causal_kernel<<<(unsigned)grid, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv
