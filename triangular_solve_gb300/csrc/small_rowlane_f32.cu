// Small-regime (m <= 64) warp-per-system launches (n <= 8) for element type float.
#include "small_launch.cuh"

namespace trsm {
int launch_rowlane_f32(const SmallArgs &a, cudaStream_t st) { return launch_rowlane_typed<float>(a, st); }
int launch_tiny_f32(const SmallArgs &a, cudaStream_t st) { return launch_tiny_typed<float>(a, st); }
}  // namespace trsm
