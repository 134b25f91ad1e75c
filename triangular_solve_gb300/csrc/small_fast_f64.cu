// Fast small-regime launches (aligned full-size systems) for element type double.
#include "small_fast.cuh"

namespace trsm {
int launch_fast_f64(const SmallArgs &a, cudaStream_t st) { return launch_fast_typed<double>(a, st); }
}  // namespace trsm
