// Unified-max (FlashDecoding++ asynchronised softmax) instantiation of the
// paged decode kernel, compiled in its own translation unit.
#include "decode_kernel.cuh"

namespace pkv {

int dispatch_decode_unified(const DecodeArgs& a, cudaStream_t stream) {
  return dispatch_decode<true>(a, stream);
}

}  // namespace pkv
