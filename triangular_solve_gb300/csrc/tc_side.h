// The f32 look-ahead form (tc_gemm.cu) with a side stream: the TF32 splits of
// each block's W-product operands (its L panel and D_b^-T), which depend on
// L and the inverted blocks only, run on a second stream one step ahead,
// beside the persistent tensor-core launch, instead of in front of the launch
// that needs them.  Events order them: a split waits for the launch that last
// read its double-buffered operands, a launch for the split it consumes, and
// the side stream starts after everything already queued on the caller's
// stream.  Every side-stream split is waited on by a later launch, so the
// caller's stream covers all of the work.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace trsm {

struct TcSide {
    cudaStream_t s = nullptr;
    cudaEvent_t launched[2] = {nullptr, nullptr}, split[2] = {nullptr, nullptr}, start = nullptr;
};

// The side stream and events of (current device, st): created by the first
// call for that pair and kept for the life of the process (no device
// memory).  The caller holds them until tc_side_release; the side stream
// starts after everything already queued on st.
int tc_side_acquire(cudaStream_t st, TcSide **side);
void tc_side_release(TcSide *side);
// tc_fused_prepare / tc_fused_step with the side stream (nullptr: none)
// tri: B is the identity (the triangular inverse); each product covers only
// the columns that can be nonzero at its step.
int tc_fused_prepare_side(int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W,
                          const float *B, int64_t ldb, void *panels, cudaStream_t st, TcSide *side, bool tri);
int tc_fused_step_side(int64_t t, int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W,
                       float *B, int64_t ldb, float alpha, void *panels, cudaStream_t st, TcSide *side, bool tri);

}  // namespace trsm
