// Fast small-regime launches (aligned full-size systems) for element type double2.
#include "small_fast.cuh"

namespace trsm {
int launch_fast_c128(const SmallArgs &a, cudaStream_t st) { return launch_fast_typed<double2>(a, st); }
}  // namespace trsm
