// Cascade (shared-prefix) decode. Placeholder until the kernel lands.
#include "internal.h"

namespace pkv {
int cascade_prefix_chunks(int, int, int, int) { return 1; }
int launch_cascade(const CascadeArgs&, cudaStream_t) { return PKV_ERR_UNSUPPORTED; }
}  // namespace pkv
