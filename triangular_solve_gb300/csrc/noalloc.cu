// trsm_llnn_noalloc: the single-system solve of trsm_llnn for callers that
// cannot allocate device memory.
//
// Who cannot allocate: code embedded in a host application that owns every
// byte of device memory through its own pool and forbids side allocations,
// and latency-sensitive paths where cudaMalloc / cudaFree (which may
// synchronise the device) are not acceptable.  This entry point calls no
// cudaMalloc, cudaFree or allocating library routine.  The blocked path's
// workspace (inverted diagonal blocks and the X_t panel) lives instead in
// the file-scope device array below, of fixed size; every GPU that loads the
// library holds that array until the process exits.
//
// Set-up: the first call on a device that reaches the blocked path looks up
// the array's device address with cudaGetSymbolAddress (with that device
// current) and caches it; make that first call before any stream capture.
// In host code the array's name is only a host-side stand-in, never a device
// address, which is why the looked-up pointer is what the kernels receive.
// The cached address belongs to the device's primary context: resetting the
// device (cudaDeviceReset) between calls is not supported.  The f32 blocked
// path also keeps one side stream and a few events per (device, caller
// stream), created by the first call that needs them (no device memory).
//
// Sharing: every call on a device uses the same array and it keeps the last
// call's contents.  Nothing in it needs to start at zero: each call writes
// every workspace element it later reads (all of W_t = D_t^{-1} including
// its zero upper blocks, and the X_t rows before they are used).  Calls whose
// work overlaps on the GPU (different streams without ordering, or several
// host threads) race on the array; serialise them.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/trsm.h"
#include "common.cuh"
#include "internal.h"

namespace {

static_assert(TRSM_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) unsigned char g_noalloc_scratch[TRSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device, then cached).
int scratch_on_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return trsm::cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return trsm::cuda_status(e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TRSM_SUCCESS;
}

int elem_size(int dtype) {
    switch (dtype) {
        case TRSM_F32: return 4;
        case TRSM_F64: return 8;
        case TRSM_C64: return 8;
        case TRSM_C128: return 16;
        default: return 0;
    }
}

bool is_zero(int dtype, const void *alpha) {
    if (dtype == TRSM_F32) return static_cast<const float *>(alpha)[0] == 0.f;
    if (dtype == TRSM_F64) return static_cast<const double *>(alpha)[0] == 0.0;
    if (dtype == TRSM_C64) {
        const float *a = static_cast<const float *>(alpha);
        return a[0] == 0.f && a[1] == 0.f;
    }
    const double *a = static_cast<const double *>(alpha);
    return a[0] == 0.0 && a[1] == 0.0;
}

bool aligned_to(const void *p, int64_t a) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)a) == 0; }

}  // namespace

extern "C" int trsm_llnn_noalloc(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha, const void *A,
                                 int64_t lda, void *B, int64_t ldb, void *stream) {
    using namespace trsm;
    const int eb = elem_size(dtype);
    if (!eb) return -1;
    if (m < 0) return -2;
    if (n < 0) return -3;
    if (!alpha) return -4;
    if (lda < (m > 1 ? m : 1)) return -6;
    if (ldb < (m > 1 ? m : 1)) return -8;
    if (m == 0 || n == 0) return TRSM_SUCCESS;
    const bool zero = is_zero(dtype, alpha);
    if (!zero && (!A || !aligned_to(A, eb))) return -5;
    if (!B || !aligned_to(B, eb)) return -7;
    if (m <= 64 && n > 64LL * 65535) return -3;

    // Only the blocked path (m > 64) reads a workspace; its size decides up
    // front whether the array can hold it: with the table's block size, else
    // with the largest smaller one that fits.
    void *scratch = nullptr;
    int64_t nb_arg = 0;  // 0: the table's block size, as trsm_llnn
    if (m > 64 && !zero) {
        const int64_t table_nb = trsm_llnn_select_nb(dtype, m, n);
        int64_t nb = table_nb;
        while (nb > 128 && blocked_workspace_bytes((int)dtype, m, n, nb) > (size_t)TRSM_NOALLOC_SCRATCH_BYTES) nb /= 2;
        if (blocked_workspace_bytes((int)dtype, m, n, nb) > (size_t)TRSM_NOALLOC_SCRATCH_BYTES)
            return TRSM_ERR_WORKSPACE;
        if (nb != table_nb) nb_arg = nb;
        const int rc = scratch_on_current_device(&scratch);
        if (rc != TRSM_SUCCESS) return rc;
    }
    // The same dispatch as trsm_llnn, with the array as the workspace and
    // allocation switched off: both entry points pick the same kernels
    // whenever the table's block size fits.
    return solve_dispatch((int)dtype, TRSM_COL_MAJOR, m, n, alpha, A, lda, 0, B, ldb, 0, 1, nb_arg, scratch,
                          scratch ? (size_t)TRSM_NOALLOC_SCRATCH_BYTES : 0, /*may_alloc=*/false,
                          static_cast<cudaStream_t>(stream), nullptr);
}
