// Small-regime (m <= 64) warp-per-system launches (n <= 8) for element type float2.
#include "small_launch.cuh"

namespace trsm {
int launch_rowlane_c64(const SmallArgs &a, cudaStream_t st) { return launch_rowlane_typed<float2>(a, st); }
int launch_tiny_c64(const SmallArgs &a, cudaStream_t st) { return launch_tiny_typed<float2>(a, st); }
}  // namespace trsm
