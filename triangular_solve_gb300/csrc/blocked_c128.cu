// Blocked-path (m > 64) driver for element type double2.
#include "blocked_launch.cuh"

namespace trsm {
int blocked_solve_c128(const BlockedArgs &a, cudaStream_t st) { return blocked_solve_typed<double2>(a, st); }
int blocked_solve_batched_c128(const BatchedBlockedArgs &a, cudaStream_t st) {
    return blocked_solve_batched_typed<double2>(a, st);
}
}  // namespace trsm
