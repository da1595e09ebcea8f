// Prefill GEMM (tensor-core path for T > 64).  Not built yet: bd_linear runs
// the decode kernel over 64-token groups until this path is available.
#include "bd_internal.h"

namespace bd {

bool prefill_available() { return false; }

cudaError_t launch_prefill(const PrefillArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace bd
