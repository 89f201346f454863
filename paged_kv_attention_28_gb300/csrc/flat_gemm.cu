// Flat GEMM of the decode phase on the sm_103a tensor cores: Y[M, N] = X[M, K] W[N, K]^T.
//
// "【FlashAttention-V4，非官方】FlashDecoding++", section 4 (Flat GEMM Optimization with
// Double Buffering), with the problem of sections 1 and 2: in decode only a few tokens
// pass through the projections at a time, so the GEMM is flat (M, the token count, is
// small; with one token it is a GEMV). Libraries pad M to 64 and waste the tensor
// cores; the page pads it to 8 and hides the memory latency with two shared-memory
// buffers, one being filled while the other is multiplied.
//
// On this hardware the GEMM is a stream of the weights W through the tensor cores:
//  * The weights are the A operand: a tile is 128 rows of W (128 output features), the
//    M of a tcgen05 kind::f16 product. The tokens are the B operand, M padded with zeros
//    to NP = 16, 32 or 64 (16 is the smallest N of a 128-row product; the TMA load fills
//    the rows past M with zeros, so nothing is written to pad). The accumulator is
//    128 TMEM lanes x NP fp32 columns.
//  * The page's two buffers become an NST-stage ring: a producer warp brings 64-column
//    slices of the W tile (16 KiB) and of X (NP x 64) by TMA into stage s while the MMA
//    warp multiplies stage s - 1, s - 2, ...; a stage is handed back when its products
//    have read it (tcgen05.commit on the stage's empty barrier).
//  * To put every SM to work on a narrow N, K is split over a thread-block cluster of
//    S CTAs (S <= 8): CTA r of the cluster multiplies its own contiguous range of K
//    slices, and the S partial tiles are summed through distributed shared memory
//    (each CTA sums a share of the rows from all S partials and writes them as bf16).
//    One launch, no workspace, and the sum is taken in a fixed order.
//
// Warps (128 threads): warp 0 TMA producer (and TMEM owner), warp 1 MMA issuer, then all
// four warps read the accumulator (warp w holds TMEM lanes 32w .. 32w + 31) for the
// reduction and the store.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();  // prefill.cu

namespace {

constexpr int FG_BM = 128;            // W rows per tile (the product's M)
constexpr int FG_BK = 64;             // K per ring stage: one 128-byte swizzled row
constexpr int FG_WSTAGE = FG_BM * FG_BK * 2;  // 16 KiB
constexpr int FG_THREADS = 128;
constexpr int FG_MAX_CLUSTER = 8;

template <int NP>
struct FgCfg {
  static constexpr int NST = NP <= 32 ? 4 : 3;         // ring stages
  static constexpr int XSTAGE = NP * FG_BK * 2;         // NP x 64 bf16
  static constexpr int SM_W = 0;
  static constexpr int SM_X = SM_W + NST * FG_WSTAGE;
  static constexpr int SM_BAR = SM_X + NST * XSTAGE;   // full[NST], empty[NST], done
  static constexpr int SM_MISC = SM_BAR + (2 * NST + 1) * 8;
  static constexpr int SMEM = SM_MISC + 16 + 1024;      // + slack to align the base to 1024
  static constexpr int TMEM_COLS = NP <= 32 ? 32 : 64;  // a power of two >= 32
  static constexpr int RED_STRIDE = NP + 4;             // floats per row of the reduction buffer
  static_assert(FG_BM * RED_STRIDE * 4 <= NST * FG_WSTAGE, "reduction buffer fits in the ring");
  static_assert(SM_X % 1024 == 0 && XSTAGE % 1024 == 0, "operand stages 1024-byte aligned");
};

struct FgArgs {
  __nv_bfloat16* y;  // [M][N]
  int32_t* err_flag;
  int m, n, k;
  int kc_per_cta;    // 64-wide K slices per CTA of a cluster
  int n_kc;          // 64-wide K slices in all
};

struct FgMisc {
  uint32_t tmem_base;
  int failed;
};

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t mbar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(mbar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Grid (S, tiles): CTA (r, t) multiplies K slices [r * kc_per_cta, ...) of W tile t, and
// the S CTAs of tile t form one cluster. Every thread reaches both cluster barriers on
// every path: the mbarrier waits are bounded, and a failed one only marks the result.
template <int NP>
__global__ void __launch_bounds__(FG_THREADS)
flat_gemm_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mx,
                 const FgArgs a) {
  using C = FgCfg<NP>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  unsigned char* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  FgMisc* misc = reinterpret_cast<FgMisc*>(smem + C::SM_MISC);
  const uint32_t bar_full = sb + C::SM_BAR, bar_empty = bar_full + 8 * C::NST,
                 bar_done = bar_empty + 8 * C::NST;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
  const int tile = blockIdx.y;
  const int kc0 = (int)rank * a.kc_per_cta;
  const int nkc = min(a.kc_per_cta, a.n_kc - kc0);  // >= 1 (the host sizes the clusters)

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    misc->failed = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&misc->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&mw);
      tma_prefetch_desc(&mx);
    }
    __syncwarp();
    const uint64_t pol = policy_evict_first();  // every weight byte is read once
    int issued = 0;
    bool ok = true;
    for (int c = 0; c < nkc; ++c) {
      const int s = c % C::NST, u = c / C::NST;
      if (u > 0 && !warp_wait(bar_empty + 8 * s, (u - 1) & 1)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        const int k0 = (kc0 + c) * FG_BK;
        mbar_arrive_expect_tx(bar_full + 8 * s, FG_WSTAGE + C::XSTAGE);
        tma_load_2d_hint(sb + C::SM_W + s * FG_WSTAGE, &mw, k0, tile * FG_BM, bar_full + 8 * s, pol);
        tma_load_2d(sb + C::SM_X + s * C::XSTAGE, &mx, k0, 0, bar_full + 8 * s);
      }
      __syncwarp();
      issued = c + 1;
    }
    if (!ok && lane == 0) {
      misc->failed = 1;
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
    // every issued copy lands before the shared memory is reused or released
    bool drained = true;
    for (int s = 0; s < C::NST && s < issued; ++s)
      if (!warp_wait(bar_full + 8 * s, ((issued - 1 - s) / C::NST) & 1)) drained = false;
    if (!drained && lane == 0) {
      misc->failed = 1;
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(FG_BM, NP, false, false);
    const uint64_t dw0 = smem_desc(sb + C::SM_W, 16, 1024, kSwizzle128B);
    const uint64_t dx0 = smem_desc(sb + C::SM_X, 16, 1024, kSwizzle128B);
    bool ok = true;
    for (int c = 0; c < nkc; ++c) {
      const int s = c % C::NST, u = c / C::NST;
      if (!warp_wait(bar_full + 8 * s, u & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dw = dw0 + (uint64_t)((s * FG_WSTAGE) >> 4);
        const uint64_t dx = dx0 + (uint64_t)((s * C::XSTAGE) >> 4);
#pragma unroll
        for (int kk = 0; kk < FG_BK / 16; ++kk)  // 16 K per product: 32 bytes along the row
          mma_bf16_ss(tmem, dw + (uint64_t)(kk * 2), dx + (uint64_t)(kk * 2), idesc, (c > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar_empty + 8 * s);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      misc->failed = 1;
      set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
    }
    // done completes once every product issued above has finished
    if (elect_one()) mma_commit(bar_done);
    __syncwarp();
  }

  // ---------------------------------------------------------------- accumulator out
  const bool done = warp_wait(bar_done, 0);
  tc_fence_after();
  if (!done && lane == 0) {
    misc->failed = 1;
    set_err(a.err_flag, PKV_DEVERR_TIMEOUT);
  }
  const int row = warp * 32 + lane;  // TMEM lane = W row within the tile
  float acc[NP];
  {
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t r[32];
    if constexpr (NP == 16) {
      tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = __uint_as_float(r[i]);
    } else {
#pragma unroll
      for (int h = 0; h < NP / 32; ++h) {
        tmem_ld32(taddr + h * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[h * 32 + i] = __uint_as_float(r[i]);
      }
    }
  }
  __syncthreads();  // every warp has read its lanes, and misc->failed is final here
  const bool failed = *reinterpret_cast<volatile int*>(&misc->failed) != 0;
  if (failed) {
#pragma unroll
    for (int i = 0; i < NP; ++i) acc[i] = NAN;
  }
  const int n0 = tile * FG_BM;
  if (S == 1) {
    const int n = n0 + row;
    if (n < a.n) {
#pragma unroll
      for (int m = 0; m < NP; ++m)
        if (m < a.m) a.y[(size_t)m * a.n + n] = __float2bfloat16_rn(acc[m]);
    }
  } else {
    // Partial tile into this CTA's reduction buffer (the ring is idle: every copy has
    // landed and every product has read it), then CTA r sums rows r, r + S, ... over
    // the S partials of the cluster, in rank order.
    float* red = reinterpret_cast<float*>(smem + C::SM_W);
#pragma unroll
    for (int i = 0; i < NP; i += 4)
      *reinterpret_cast<float4*>(red + row * C::RED_STRIDE + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    cluster_sync_all();
    constexpr int G4 = NP / 4;  // float4 groups per row
    const int my_rows = (FG_BM - (int)rank + S - 1) / S;
    const uint32_t red_addr = smem_u32(red);
    for (int it = threadIdx.x; it < my_rows * G4; it += FG_THREADS) {
      const int rr = (int)rank + S * (it / G4);
      const int m0 = (it % G4) * 4;
      const uint32_t off = red_addr + (uint32_t)((rr * C::RED_STRIDE + m0) * 4);
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < S; ++q) {
        const float4 v = ld_cluster_f4(map_shared_rank(off, (uint32_t)q));
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
      }
      const int n = n0 + rr;
      if (n < a.n) {
        const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (m0 + j < a.m) a.y[(size_t)(m0 + j) * a.n + n] = __float2bfloat16_rn(vals[j]);
      }
    }
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while another still reads its buffer
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

bool encode_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)FG_BK, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NP>
int launch_fg(const FlatGemmArgs& p, const FlatGemmPlan& plan, cudaStream_t stream) {
  using C = FgCfg<NP>;
  CUtensorMap mw, mx;
  // W [N][K]: boxes of 128 rows x 64 columns; X [M][K]: NP rows (rows past M read as 0)
  if (!encode_bf16_2d(&mw, p.w, (uint64_t)p.k, (uint64_t)p.n, FG_BM) ||
      !encode_bf16_2d(&mx, p.x, (uint64_t)p.k, (uint64_t)p.m, NP))
    return check_launch(cudaErrorInvalidValue);
  static FuncConfigured configured;
  if (!configured.ensure(reinterpret_cast<const void*>(flat_gemm_kernel<NP>), C::SMEM)) return PKV_ERR_LAUNCH;
  FgArgs a{static_cast<__nv_bfloat16*>(p.y), p.err_flag, p.m, p.n, p.k, plan.kc_per_cta, plan.n_kc};
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)plan.splits, (unsigned)plan.tiles, 1);
  cfg.blockDim = dim3(FG_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)plan.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return check_launch(cudaLaunchKernelEx(&cfg, flat_gemm_kernel<NP>, mw, mx, a));
}

}  // namespace

int flat_gemm_padded_m(int m) { return m <= 16 ? 16 : m <= 32 ? 32 : 64; }

// Tiles of 128 W rows, and K split over a cluster of S CTAs per tile: the largest S <= 8
// for which every CTA of the grid is resident at once (tiles x S <= SMs x CTAs per SM),
// then S trimmed so that every CTA gets at least one 64-column slice of K.
FlatGemmPlan plan_flat_gemm(int m, int n, int k) {
  FlatGemmPlan p{};
  p.tiles = (n + FG_BM - 1) / FG_BM;
  p.n_kc = (k + FG_BK - 1) / FG_BK;
  const int np = flat_gemm_padded_m(m);
  const int smem = np == 16 ? FgCfg<16>::SMEM : np == 32 ? FgCfg<32>::SMEM : FgCfg<64>::SMEM;
  int sms = device_sm_count();
  if (sms <= 0) sms = 148;
  int per_sm = (228 * 1024) / (smem + 1024);
  if (per_sm < 1) per_sm = 1;
  const long slots = (long)sms * per_sm;
  long s = slots / p.tiles;
  if (s > FG_MAX_CLUSTER) s = FG_MAX_CLUSTER;
  if (s > p.n_kc) s = p.n_kc;
  if (s < 1) s = 1;
  p.kc_per_cta = (p.n_kc + (int)s - 1) / (int)s;
  p.splits = (p.n_kc + p.kc_per_cta - 1) / p.kc_per_cta;
  return p;
}

int launch_flat_gemm(const FlatGemmArgs& a, cudaStream_t stream) {
  const FlatGemmPlan plan = plan_flat_gemm(a.m, a.n, a.k);
  if (plan.tiles > 65535) return PKV_ERR_UNSUPPORTED;
  switch (flat_gemm_padded_m(a.m)) {
    case 16: return launch_fg<16>(a, plan, stream);
    case 32: return launch_fg<32>(a, plan, stream);
    default: return launch_fg<64>(a, plan, stream);
  }
}

}  // namespace pkv
