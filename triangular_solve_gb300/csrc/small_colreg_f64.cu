// Small-regime (m <= 64) thread-per-column launches for element type double,
// and the alpha == 0 fill.
#include "small_launch.cuh"

namespace trsm {
int launch_colreg_f64(const SmallArgs &a, cudaStream_t st) { return launch_colreg_typed<double>(a, st); }
int launch_zero_f64(const SmallArgs &a, cudaStream_t st) { return launch_zero_typed<double>(a, st); }
}  // namespace trsm
