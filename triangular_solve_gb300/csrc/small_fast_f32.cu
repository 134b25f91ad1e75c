// Fast small-regime launches (aligned full-size systems) for element type float.
#include "small_fast.cuh"

namespace trsm {
int launch_fast_f32(const SmallArgs &a, cudaStream_t st) { return launch_fast_typed<float>(a, st); }
}  // namespace trsm
