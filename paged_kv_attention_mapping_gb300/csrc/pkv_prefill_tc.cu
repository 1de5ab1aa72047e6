// Tensor-core prefill-chunk attention (tcgen05 / TMEM) — not built yet: every
// row goes through the row path.
#include "pkv_internal.h"

namespace pkv {

bool prefill_tc_supported(int, int, int) { return false; }

cudaError_t launch_prefill_tc(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pkv
