// Blocked-path (m > 64) driver for element type double.
#include "blocked_launch.cuh"

namespace trsm {
int blocked_solve_f64(const BlockedArgs &a, cudaStream_t st) { return blocked_solve_typed<double>(a, st); }
int blocked_solve_batched_f64(const BatchedBlockedArgs &a, cudaStream_t st) {
    return blocked_solve_batched_typed<double>(a, st);
}
}  // namespace trsm
