// Paged decode over FP8 E4M3 page pools (bf16 query and output), compiled in its own
// translation unit. FP8 is named as a way to cut attention's memory traffic in
// "TensorRT-LLM深度优化：利用FMHA（Fused Multi-Head Attention）内核加速Hopper架构推理",
// section 4; the E4M3 format and the per-(page, KV head) scales are this library's reading.
#include "decode_kernel.cuh"

namespace pkv {

int dispatch_decode_fp8(const DecodeArgs& a, cudaStream_t stream) {
  const int G = a.n_qo_heads / a.n_kv_heads;
  // a CTA takes two adjacent KV heads (one copy moves both heads' tiles of a page)
  if (a.page_size != 16 || a.dtype != PKV_BF16 || a.unified || a.n_kv_heads % 2) return PKV_ERR_UNSUPPORTED;
#define PKV_FP8_CASE(DD, GG) \
  if (a.head_dim == DD && G == GG) return launch_decode_t<__nv_bfloat16, DD, 16, GG, false, true>(a, stream);
  PKV_FP8_CASE(64, 1) PKV_FP8_CASE(64, 2) PKV_FP8_CASE(64, 4) PKV_FP8_CASE(64, 8)
  PKV_FP8_CASE(128, 1) PKV_FP8_CASE(128, 2) PKV_FP8_CASE(128, 4) PKV_FP8_CASE(128, 8)
#undef PKV_FP8_CASE
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
