// Small-regime (m <= 64) warp-per-system launches (n <= 8) for element type double.
#include "small_launch.cuh"

namespace trsm {
int launch_rowlane_f64(const SmallArgs &a, cudaStream_t st) { return launch_rowlane_typed<double>(a, st); }
int launch_tiny_f64(const SmallArgs &a, cudaStream_t st) { return launch_tiny_typed<double>(a, st); }
}  // namespace trsm
