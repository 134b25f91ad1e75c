// Blocked-path (m > 64) driver for element type float.
#include "blocked_launch.cuh"

namespace trsm {
int blocked_solve_f32(const BlockedArgs &a, cudaStream_t st) { return blocked_solve_typed<float>(a, st); }
int blocked_solve_batched_f32(const BatchedBlockedArgs &a, cudaStream_t st) {
    return blocked_solve_batched_typed<float>(a, st);
}
}  // namespace trsm
