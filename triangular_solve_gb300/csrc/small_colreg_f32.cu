// Small-regime (m <= 64) thread-per-column launches for element type float,
// and the alpha == 0 fill.
#include "small_launch.cuh"

namespace trsm {
int launch_colreg_f32(const SmallArgs &a, cudaStream_t st) {
    const int rc = launch_fast_f32(a, st);
    return rc == -100000 ? launch_colreg_typed<float>(a, st) : rc;
}
int launch_zero_f32(const SmallArgs &a, cudaStream_t st) { return launch_zero_typed<float>(a, st); }
}  // namespace trsm
