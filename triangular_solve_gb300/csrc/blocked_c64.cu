// Blocked-path (m > 64) driver for element type float2.
#include "blocked_launch.cuh"

namespace trsm {
int blocked_solve_c64(const BlockedArgs &a, cudaStream_t st) { return blocked_solve_typed<float2>(a, st); }
int blocked_solve_batched_c64(const BatchedBlockedArgs &a, cudaStream_t st) {
    return blocked_solve_batched_typed<float2>(a, st);
}
}  // namespace trsm
