// Fast small-regime launches (aligned full-size systems) for element type float2.
#include "small_fast.cuh"

namespace trsm {
int launch_fast_c64(const SmallArgs &a, cudaStream_t st) { return launch_fast_typed<float2>(a, st); }
}  // namespace trsm
