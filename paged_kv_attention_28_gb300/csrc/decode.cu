// Online-softmax paged decode, the split merge, and the pairwise state merge.
#include "decode_kernel.cuh"
#include "merge.cuh"

namespace pkv {

// Combines the live splits of each (sequence, query head) row by log-sum-exp, one CTA of
// kMergeWarps warps per row (merge_row_cta): with up to 8 kMergeWarps splits every load of
// the row is in flight at once, so a row costs about one round trip to L2, where the
// decode kernel's partial states still are. Rows whose sequence fits in one split were
// written by the decode kernel and are skipped here.
constexpr int kMergeWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_splits_kernel(const DecodeArgs a) {
  __shared__ float sm[kMergeWarps * (D + 3)];
  const int row = blockIdx.x;
  const int b = row / a.n_qo_heads;
  const int P = a.page_size;
  const int L = __ldg(a.kv_lens + b);  // an input of the decode kernel, not one of its results
  // Launched as a programmatic dependent of the decode kernel: wait until that grid has
  // finished and its partial states are visible. Every CTA waits, so that this grid never
  // ends before the decode grid.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (L < 0 || L > a.max_blocks * P) return;  // the decode kernel wrote NaN
  const int nblk = (L + P - 1) / P;
  const int n_live = (nblk + a.pages_per_split - 1) / a.pages_per_split;
  if (n_live < 2) return;
  const float* pl = a.part_lse + (size_t)row * a.num_splits;
  const float* po = a.part_o + (size_t)row * a.num_splits * D;
  merge_row_cta<T, D, kMergeWarps>(
      n_live, [&](int i) { return __ldcg(pl + i); }, [&](int i) { return po + (size_t)i * D; },
      static_cast<T*>(a.out) + (size_t)row * D, a.lse ? a.lse + row : nullptr, sm);
}

template <typename T, int D>
int launch_merge_t(const DecodeArgs& a, cudaStream_t stream) {
  const int rows = a.batch * a.n_qo_heads;
  // Programmatic dependent launch: the merge's CTAs are placed while the decode grid's last
  // CTAs still run, and read each row's sequence length before the decode grid ends.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)rows, 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return check_launch(cudaLaunchKernelEx(&cfg, merge_splits_kernel<T, D>, a));
}

int launch_merge_splits(const DecodeArgs& a, cudaStream_t stream) {
  if (a.dtype == PKV_F32) {
    if (a.head_dim == 64) return launch_merge_t<float, 64>(a, stream);
    if (a.head_dim == 128) return launch_merge_t<float, 128>(a, stream);
  } else {
    if (a.head_dim == 64) return launch_merge_t<__nv_bfloat16, 64>(a, stream);
    if (a.head_dim == 128) return launch_merge_t<__nv_bfloat16, 128>(a, stream);
  }
  return PKV_ERR_UNSUPPORTED;
}

int dispatch_decode_unified(const DecodeArgs& a, cudaStream_t stream);  // decode_um.cu
int dispatch_decode_fp8(const DecodeArgs& a, cudaStream_t stream);      // decode_fp8.cu

int decode_ctas_per_sm(int dtype, int head_dim, int group) {
#define PKV_CPS(TT, F8)                                                        \
  if (head_dim == 64) {                                                        \
    if (group == 1) return ctas_per_sm_t<TT, 64, 1, F8>();                     \
    if (group == 2) return ctas_per_sm_t<TT, 64, 2, F8>();                     \
    if (group == 4) return ctas_per_sm_t<TT, 64, 4, F8>();                     \
    if (group == 8) return ctas_per_sm_t<TT, 64, 8, F8>();                     \
  } else {                                                                     \
    if (group == 1) return ctas_per_sm_t<TT, 128, 1, F8>();                    \
    if (group == 2) return ctas_per_sm_t<TT, 128, 2, F8>();                    \
    if (group == 4) return ctas_per_sm_t<TT, 128, 4, F8>();                    \
    if (group == 8) return ctas_per_sm_t<TT, 128, 8, F8>();                    \
  }
  if (dtype == PKV_F32) {
    PKV_CPS(float, false)
  } else if (dtype == PKV_FP8_E4M3) {
    PKV_CPS(__nv_bfloat16, true)
  } else {
    PKV_CPS(__nv_bfloat16, false)
  }
#undef PKV_CPS
  return 2;
}

bool decode_supported(int dtype, int head_dim, int page_size, int group) {
  return (dtype == PKV_F32 || dtype == PKV_BF16) && (head_dim == 64 || head_dim == 128) &&
         page_size == 16 && (group == 1 || group == 2 || group == 4 || group == 8);
}

int launch_decode_partials(const DecodeArgs& a, cudaStream_t stream) {
  if (decode_tc_supported(a)) return launch_decode_tc(a, stream);
  return a.unified ? dispatch_decode_unified(a, stream) : dispatch_decode<false>(a, stream);
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const int rc = decode_tc_supported(a) ? launch_decode_tc(a, stream)
                 : a.fp8                  ? dispatch_decode_fp8(a, stream)
                 : a.unified              ? dispatch_decode_unified(a, stream)
                                          : dispatch_decode<false>(a, stream);
  if (rc != PKV_OK) return rc;
  if (a.num_splits > 1) return launch_merge_splits(a, stream);
  return PKV_OK;
}

// ------------------------------------------------------------------ pairwise merge

template <typename T>
__global__ void __launch_bounds__(128)
merge_pair_kernel(const float* oa, const float* la, const float* ob,
                  const float* lb, T* out, float* lse, int n_rows, int D) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const float a = la[row];
  const float bb = lb[row];
  __syncwarp();  // every lane has read lse before lane 0 may overwrite it in place
  const float M = fmaxf(a, bb);
  const bool empty = (M == -INFINITY);
  const float wa = empty ? 0.0f : ex2((a - M) * kLog2e);
  const float wb = empty ? 0.0f : ex2((bb - M) * kLog2e);
  const float inv = empty ? 0.0f : 1.0f / (wa + wb);
  for (int d = lane; d < D; d += 32) {
    const size_t i = (size_t)row * D + d;
    const float x = empty ? 0.0f : (wa * oa[i] + wb * ob[i]) * inv;
    out[i] = from_f32<T>(x);
  }
  if (lse && lane == 0) lse[row] = empty ? -INFINITY : M + logf(wa + wb);
}

int launch_merge_pair(const float* out_a, const float* lse_a, const float* out_b,
                      const float* lse_b, void* out, float* lse, int n_rows, int head_dim,
                      int out_dtype, cudaStream_t stream) {
  if (n_rows == 0) return PKV_OK;
  const int grid = (n_rows + 3) / 4;
  if (out_dtype == PKV_F32)
    merge_pair_kernel<float><<<grid, 128, 0, stream>>>(out_a, lse_a, out_b, lse_b,
                                                      static_cast<float*>(out), lse, n_rows, head_dim);
  else
    merge_pair_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(
        out_a, lse_a, out_b, lse_b, static_cast<__nv_bfloat16*>(out), lse, n_rows, head_dim);
  return check_launch(cudaGetLastError());
}

}  // namespace pkv
