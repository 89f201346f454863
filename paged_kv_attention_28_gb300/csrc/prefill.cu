// Causal prefill (tcgen05 + TMEM + TMA). Placeholder until the kernel lands.
#include "internal.h"

namespace pkv {
int launch_prefill(const PrefillArgs&, cudaStream_t) { return PKV_ERR_UNSUPPORTED; }
}  // namespace pkv
