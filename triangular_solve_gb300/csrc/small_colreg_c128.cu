// Small-regime (m <= 64) thread-per-column launches for element type double2,
// and the alpha == 0 fill.
#include "small_launch.cuh"

namespace trsm {
int launch_colreg_c128(const SmallArgs &a, cudaStream_t st) {
    const int rc = launch_fast_c128(a, st);
    return rc == -100000 ? launch_colreg_typed<double2>(a, st) : rc;
}
int launch_zero_c128(const SmallArgs &a, cudaStream_t st) { return launch_zero_typed<double2>(a, st); }
}  // namespace trsm
