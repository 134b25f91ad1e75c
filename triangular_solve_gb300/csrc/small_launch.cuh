// Host-side launch of the small-regime kernels for one element type.
#pragma once

#include "internal.h"
#include "small_kernels.cuh"

namespace trsm {

// Registers per thread bound the row chunk: a thread keeps RC elements of its
// column live.  Complex double keeps at most 32 (64 doubles) in chunks that
// divide M; the other types keep the whole column.
template <typename T, int M>
constexpr int small_rc() {
    return (sizeof(T) >= 16 && M > 32) ? (M % 32 == 0 ? 32 : M / 2) : M;
}
static_assert(64 % small_rc<double2, 64>() == 0 && 48 % small_rc<double2, 48>() == 0, "chunks divide M");

template <typename Kern>
static int set_smem(Kern k, size_t bytes) {
    if (bytes > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return TRSM_SUCCESS;
}

template <typename T, int M, int NC>
static int launch_rowlane(SmallGeom g, T alpha, cudaStream_t st) {
    g.spc = 4;
    g.w = NC;
    const size_t smem = (size_t)g.spc * SmallImage<T, M>::elems(NC) * sizeof(T);
    auto kern = small_rowlane_kernel<T, M, NC>;
    int rc = set_smem(kern, smem);
    if (rc) return rc;
    const dim3 grid((unsigned)((g.batch + g.spc - 1) / g.spc));
    kern<<<grid, 32 * g.spc, smem, st>>>(g, alpha);
    return launch_status();
}

// Columns spread over CTAs: one warp per (system, NC-column slice).  For
// FP64 batches too small to fill the GPU with whole systems, where a system
// on one SM would be bound by that SM's FP64 rate.
template <typename T, int M, int NC>
static int launch_rowlane_split(SmallGeom g, T alpha, cudaStream_t st) {
    g.spc = 1;
    g.w = NC;
    const size_t smem = SmallImage<T, M>::elems(NC) * sizeof(T);
    auto kern = small_rowlane_kernel<T, M, NC>;
    int rc = set_smem(kern, smem);
    if (rc) return rc;
    const dim3 grid((unsigned)g.batch, (unsigned)((g.n + NC - 1) / NC));
    kern<<<grid, 32, smem, st>>>(g, alpha);
    return launch_status();
}

// NC as large as keeps at least two CTAs per SM (else 1).
template <typename T, int M>
static int launch_rowlane_split_m(const SmallGeom &g, T alpha, int sms, cudaStream_t st) {
    auto slices = [&](int nc) { return g.batch * ((g.n + nc - 1) / nc); };
    if (slices(8) >= 2 * sms) return launch_rowlane_split<T, M, 8>(g, alpha, st);
    if (slices(4) >= 2 * sms) return launch_rowlane_split<T, M, 4>(g, alpha, st);
    if (slices(2) >= 2 * sms) return launch_rowlane_split<T, M, 2>(g, alpha, st);
    return launch_rowlane_split<T, M, 1>(g, alpha, st);
}

template <typename T, int M>
static int launch_colreg_m(SmallGeom g, T alpha, cudaStream_t st) {
    const int w = g.n < 64 ? g.n : 64;
    const size_t per = (size_t)SmallImage<T, M>::elems(w) * sizeof(T);
    int spc = 128 / w > 1 ? 128 / w : 1;
    while (spc > 1 && (size_t)spc * per > 225 * 1024) --spc;
    g.spc = spc;
    g.w = w;
    const size_t smem = (size_t)spc * per;
    auto kern = small_colreg_kernel<T, M, small_rc<T, M>()>;
    int rc = set_smem(kern, smem);
    if (rc) return rc;
    const dim3 grid((unsigned)((g.batch + spc - 1) / spc), (unsigned)((g.n + w - 1) / w));
    kern<<<grid, spc * w, smem, st>>>(g, alpha);
    return launch_status();
}

template <typename T, int M>
static int launch_rowlane_m(SmallGeom g, T alpha, cudaStream_t st) {
    if (g.n <= 1) return launch_rowlane<T, M, 1>(g, alpha, st);
    if (g.n <= 2) return launch_rowlane<T, M, 2>(g, alpha, st);
    if (g.n <= 4) return launch_rowlane<T, M, 4>(g, alpha, st);
    return launch_rowlane<T, M, 8>(g, alpha, st);
}

inline SmallGeom small_geom(const SmallArgs &a) {
    SmallGeom g;
    g.m = (int)a.m;
    g.n = (int)a.n;
    g.layout = a.layout;
    g.A = a.A;
    g.lda = a.lda;
    g.sA = a.strideA;
    g.B = a.B;
    g.ldb = a.ldb;
    g.sB = a.strideB;
    g.batch = a.batch;
    g.spc = 1;
    g.w = 1;
    return g;
}

// m <= 8: a thread per (system, column).
template <typename T>
int launch_tiny_typed(const SmallArgs &a, cudaStream_t st) {
    const SmallGeom g = small_geom(a);
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    const int64_t threads = g.batch * g.n;
    small_tiny_kernel<T><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(g, alpha);
    return launch_status();
}

// Thread-per-column kernel (n > 8).
template <typename T>
int launch_colreg_typed(const SmallArgs &a, cudaStream_t st) {
    const SmallGeom g = small_geom(a);
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    if (g.m <= 8) return launch_colreg_m<T, 8>(g, alpha, st);
    if (g.m <= 16) return launch_colreg_m<T, 16>(g, alpha, st);
    if (g.m <= 32) return launch_colreg_m<T, 32>(g, alpha, st);
    if (g.m <= 48) return launch_colreg_m<T, 48>(g, alpha, st);
    return launch_colreg_m<T, 64>(g, alpha, st);
}

// Warp-per-system kernel (n <= 8).
template <typename T>
int launch_rowlane_typed(const SmallArgs &a, cudaStream_t st) {
    const SmallGeom g = small_geom(a);
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    if (g.m <= 8) return launch_rowlane_m<T, 8>(g, alpha, st);
    if (g.m <= 16) return launch_rowlane_m<T, 16>(g, alpha, st);
    if (g.m <= 32) return launch_rowlane_m<T, 32>(g, alpha, st);
    if (g.m <= 48) return launch_rowlane_m<T, 48>(g, alpha, st);
    return launch_rowlane_m<T, 64>(g, alpha, st);
}

template <typename T>
int launch_zero_typed(const SmallArgs &a, cudaStream_t st) {
    const int64_t total = a.m * a.n * a.batch;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    zero_rhs_kernel<T><<<(unsigned)blocks, threads, 0, st>>>(static_cast<T *>(a.B), a.m, a.n, a.ldb, a.strideB,
                                                             a.batch, a.layout);
    return launch_status();
}

}  // namespace trsm
