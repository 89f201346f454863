// attn_decode_paged_noalloc: paged decode whose split partial states live in a
// fixed scratch array that belongs to the library. The caller passes no workspace,
// and the call allocates no device memory.
#include <cuda.h>

#include <mutex>

#include "internal.h"

namespace pkv {
namespace {

// One scratch area per device that loads the library. It holds the fp32 partial
// (O, LSE) states of split decode and stays allocated until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Host code cannot use g_decode_scratch directly: in host code that name is a
// host-side stand-in, not a device address. The device address is looked up with the
// device current and cached per device together with the id of the context it belongs
// to. A context that replaces the old one (after cudaDeviceReset, say) has another id,
// and its module's copy of the array another address, so the lookup is made again.
constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchSlot g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current context (false when there is none or the
// driver does not say).
bool current_context_id(unsigned long long* id) {
  static const PfnCtxGetCurrent get_current = []() -> PfnCtxGetCurrent {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<PfnCtxGetCurrent>(p)
               : nullptr;
  }();
  static const PfnCtxGetId get_id = []() -> PfnCtxGetId {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<PfnCtxGetId>(p)
               : nullptr;
  }();
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_DEVICE;
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& slot = g_scratch[dev];
  if (!have_id || !slot.ptr || slot.ctx_id != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) return check_launch(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
    // Without a context id the address is not kept: it is looked up on every call.
    slot.ptr = have_id ? p : nullptr;
    slot.ctx_id = id;
    *out = p;
    return PKV_OK;
  }
  *out = slot.ptr;
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int attn_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                         const int32_t* block_table, const int32_t* kv_lens,
                                         void* out, float* lse, int batch, int max_blocks_per_seq,
                                         int num_pages, int n_qo_heads, int n_kv_heads,
                                         int head_dim, int page_size, float scale, int num_splits,
                                         int dtype, int32_t* err_flag, void* stream) {
  const size_t need = attn_decode_workspace_size(batch, max_blocks_per_seq, n_qo_heads, n_kv_heads,
                                                 head_dim, page_size, num_splits, dtype);
  if (need == (size_t)-1) return PKV_ERR_INVALID_ARG;
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = pkv::scratch_for_current_device(&scratch);
    if (rc != PKV_OK) return rc;
  }
  return attn_decode_paged(q, k_pages, v_pages, block_table, kv_lens, out, lse, batch,
                           max_blocks_per_seq, num_pages, n_qo_heads, n_kv_heads, head_dim,
                           page_size, scale, num_splits, dtype, scratch,
                           need > 0 ? (size_t)PKV_NOALLOC_SCRATCH_BYTES : 0, err_flag, stream);
}
