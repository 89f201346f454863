// Work distribution for kernels whose grid has one CTA per work item but keeps only one
// CTA per SM resident: a running CTA takes further items by cancelling CTAs of its own
// grid that have not started yet (Blackwell cluster launch control). The hardware hands
// out the pending CTAs in launch order, so items go, in index order, to whichever CTA
// asks first, i.e. to the first one to run short of work.
//
// Item 0 of a CTA is its own blockIdx.x. During item k one warp asks for item k + 1; the
// response lands in ring slot k % NXS. Every warp reads it when it reaches the end of
// item k and then arrives on that slot's next_empty barrier; a failed response (no
// pending CTA left) ends every warp's loop, and no request follows it.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace pkv {

constexpr int NXS = 4;  // slots of the response ring

__device__ __forceinline__ void request_next_cta(uint32_t slot, uint32_t full) {
  mbar_arrive_expect_tx(full, 16);
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
          slot),
      "r"(full)
      : "memory");
}

// The index of the CTA that a response cancelled, or -1 if it cancelled none.
__device__ __forceinline__ int response_cta(uint32_t slot) {
  int x;
  asm volatile(
      "{\n\t.reg .b128 rr;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 rr, [%1];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, rr;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, rr;\n\t"
      "@!p mov.b32 %0, -1;\n\t}"
      : "=r"(x)
      : "r"(slot)
      : "memory");
  return x;
}

// Where the ring lives: the responses, next_full[0] and next_empty[0] (consecutive).
struct NextRing {
  uint32_t slot0, full0, empty0;
};

// Item k + 1 of this CTA, read by a whole warp at the end of its item k; n_items if
// there is none (or if the response never came, which is reported).
__device__ __forceinline__ int next_item(const NextRing& ring, uint32_t k, int n_items, int32_t* err) {
  const uint32_t s = k % NXS, u = k / NXS;
  int id = n_items;
  if (warp_wait(ring.full0 + 8 * s, u & 1)) {
    const int x = response_cta(ring.slot0 + 16 * s);
    if (x >= 0 && x < n_items) id = x;
  } else if ((threadIdx.x & 31) == 0) {
    set_err(err, PKV_DEVERR_TIMEOUT);
  }
  __syncwarp();
  if (elect_one()) mbar_arrive(ring.empty0 + 8 * s);
  __syncwarp();
  return id;
}

}  // namespace pkv
