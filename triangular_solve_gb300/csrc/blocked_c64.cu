// Blocked-path (m > 64) driver for element type float2.
#include "blocked_launch.cuh"

namespace trsm {
int blocked_solve_c64(const BlockedArgs &a, cudaStream_t st) { return blocked_solve_typed<float2>(a, st); }
}  // namespace trsm
