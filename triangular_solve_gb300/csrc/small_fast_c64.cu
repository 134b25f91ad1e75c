// Fast small-regime launches (aligned full-size systems) for element type float2:
// the TMA-streaming kernel for batches of m = 32, 48, 64 systems, else the
// chunked kernel.
#include "small_tma_c64.cuh"

namespace trsm {
int launch_fast_c64(const SmallArgs &a, cudaStream_t st) {
    const int rc = launch_tma_c64(a, st);
    if (rc != kTmaNotApplicable) return rc;
    return launch_fast_typed<float2>(a, st);
}
}  // namespace trsm
