// C ABI of the GB300 triangular-solve library: argument checking, path
// selection (small regime for m <= 64, blocked path above), workspace
// handling and the row-major adapter.  See include/trsm.h for the contract.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include <cuda_runtime.h>

#include "../../include/trsm.h"
#include "blocked_kernels.cuh"
#include "internal.h"
#include "nb_table.h"

using namespace trsm;

namespace {

int elem_bytes(int dtype) {
    switch (dtype) {
        case TRSM_F32: return 4;
        case TRSM_F64: return 8;
        case TRSM_C64: return 8;
        case TRSM_C128: return 16;
        default: return 0;
    }
}

bool alpha_is_zero(int dtype, const void *alpha) {
    switch (dtype) {
        case TRSM_F32: return static_cast<const float *>(alpha)[0] == 0.f;
        case TRSM_F64: return static_cast<const double *>(alpha)[0] == 0.0;
        case TRSM_C64: {
            const float *a = static_cast<const float *>(alpha);
            return a[0] == 0.f && a[1] == 0.f;
        }
        default: {
            const double *a = static_cast<const double *>(alpha);
            return a[0] == 0.0 && a[1] == 0.0;
        }
    }
}

bool aligned(const void *p, int64_t a) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)a) == 0; }

int64_t max1(int64_t x) { return x > 1 ? x : 1; }

int nearest_nb(int dtype, int64_t m) {
    int best = 0;
    double best_d = 1e300;
    for (const NbEntry &e : kNbTable) {
        if (e.dtype != dtype) continue;
        const double d = fabs(log2((double)m) - log2((double)e.m));
        if (d < best_d) {
            best_d = d;
            best = e.nb;
        }
    }
    return best ? best : 256;
}

constexpr int kFastNotApplicableCode = -100000;  // launch_fast_*: preconditions not met

int launch_small(int dtype, const SmallArgs &a, cudaStream_t st) {
    if (a.m <= 8 && a.batch * a.n <= (int64_t)256 * 0x7fffffff) {
        switch (dtype) {
            case TRSM_F32: return launch_tiny_f32(a, st);
            case TRSM_F64: return launch_tiny_f64(a, st);
            case TRSM_C64: return launch_tiny_c64(a, st);
            default: return launch_tiny_c128(a, st);
        }
    }
    if (a.n <= 8) {
        switch (dtype) {
            case TRSM_F32: return launch_rowlane_f32(a, st);
            case TRSM_F64: return launch_rowlane_f64(a, st);
            case TRSM_C64: return launch_rowlane_c64(a, st);
            default: return launch_rowlane_c128(a, st);
        }
    }
    switch (dtype) {
        case TRSM_F32: return launch_colreg_f32(a, st);
        case TRSM_F64: return launch_colreg_f64(a, st);
        case TRSM_C64: return launch_colreg_c64(a, st);
        default: return launch_colreg_c128(a, st);
    }
}

int launch_zero(int dtype, const SmallArgs &a, cudaStream_t st) {
    switch (dtype) {
        case TRSM_F32: return launch_zero_f32(a, st);
        case TRSM_F64: return launch_zero_f64(a, st);
        case TRSM_C64: return launch_zero_c64(a, st);
        default: return launch_zero_c128(a, st);
    }
}

int blocked_solve(int dtype, const BlockedArgs &a, cudaStream_t st) {
    switch (dtype) {
        case TRSM_F32: return blocked_solve_f32(a, st);
        case TRSM_F64: return blocked_solve_f64(a, st);
        case TRSM_C64: return blocked_solve_c64(a, st);
        default: return blocked_solve_c128(a, st);
    }
}

int blocked_solve_batched(int dtype, const BatchedBlockedArgs &a, cudaStream_t st) {
    switch (dtype) {
        case TRSM_F32: return blocked_solve_batched_f32(a, st);
        case TRSM_F64: return blocked_solve_batched_f64(a, st);
        case TRSM_C64: return blocked_solve_batched_c64(a, st);
        default: return blocked_solve_batched_c128(a, st);
    }
}

// Batches of systems up to this order run the blocked path over the whole
// batch in one launch sequence (FMA-pipe products); larger systems run it
// system by system, where each system alone fills the GPU.
constexpr int64_t kBatchedMaxM = 2048;
// Upper bound of one chunk's workspace: larger batches run chunk by chunk.
constexpr size_t kBatchedChunkBytes = size_t(1) << 30;

// Batch of m > 64 systems through the batched blocked path, in chunks of at
// most 65535 systems and kBatchedChunkBytes of workspace.  Row-major systems
// are solved on column-major copies in the workspace.
int solve_batched(int dtype, int layout, int64_t m, int64_t n, const unsigned char *alpha, const void *A,
                  int64_t lda, int64_t sA, void *B, int64_t ldb, int64_t sB, int64_t batch, int64_t nb, void *ws,
                  size_t ws_bytes, bool may_alloc, cudaStream_t st) {
    const int eb = elem_bytes(dtype);
    const bool shared = sA == 0;
    const bool row = layout == TRSM_ROW_MAJOR;
    auto chunk_bytes = [&](int64_t c, size_t *a_off, size_t *b_off) {
        size_t b = batched_workspace_bytes(dtype, m, n, nb, c, shared);
        *a_off = b;
        if (row) b += (size_t)round256((shared ? 1 : c) * m * m * eb);
        *b_off = b;
        if (row) b += (size_t)round256(c * m * n * eb);
        return b;
    };
    size_t ao = 0, bo = 0;
    const size_t per = chunk_bytes(1, &ao, &bo);
    int64_t cnt = (int64_t)(kBatchedChunkBytes / (per ? per : 1));
    if (cnt < 1) cnt = 1;
    if (cnt > batch) cnt = batch;
    if (cnt > 65535) cnt = 65535;
    const size_t total = chunk_bytes(cnt, &ao, &bo);
    void *mem = ws;
    bool owned = false;
    if (mem == nullptr || ws_bytes < total) {
        if (!may_alloc) return TRSM_ERR_WORKSPACE;
        const int ae = workspace_alloc(&mem, total, st);
        if (ae) return ae;
        owned = true;
    }
    int rc = TRSM_SUCCESS;
    for (int64_t b0 = 0; b0 < batch && rc == TRSM_SUCCESS; b0 += cnt) {
        const int64_t c = batch - b0 < cnt ? batch - b0 : cnt;
        const char *Ab = static_cast<const char *>(A) + b0 * sA * eb;
        char *Bb = static_cast<char *>(B) + b0 * sB * eb;
        BatchedBlockedArgs ba;
        ba.m = m; ba.n = n; ba.nb = nb;
        ba.batch = c;
        ba.ws = mem;
        memcpy(ba.alpha, alpha, sizeof(ba.alpha));
        if (!row) {
            ba.A = Ab; ba.lda = lda; ba.strideA = sA;
            ba.B = Bb; ba.ldb = ldb; ba.strideB = sB;
            rc = blocked_solve_batched(dtype, ba, st);
        } else {
            char *Lc = static_cast<char *>(mem) + ao;
            char *Bc = static_cast<char *>(mem) + bo;
            rc = launch_transpose_copy(eb, Ab, lda, Lc, m, m, m, st, sA, m * m, shared ? 1 : (int)c);
            if (!rc) rc = launch_transpose_copy(eb, Bb, ldb, Bc, m, m, n, st, sB, m * n, (int)c);
            ba.A = Lc; ba.lda = m; ba.strideA = shared ? 0 : m * m;
            ba.B = Bc; ba.ldb = m; ba.strideB = m * n;
            if (!rc) rc = blocked_solve_batched(dtype, ba, st);
            if (!rc) rc = launch_transpose_copy(eb, Bc, m, Bb, ldb, n, m, st, m * n, sB, (int)c);
        }
    }
    if (owned) {
        const cudaError_t e = cudaFreeAsync(mem, st);
        if (rc == TRSM_SUCCESS && e != cudaSuccess) rc = cuda_status(e);
    }
    return rc;
}

}  // namespace

namespace trsm {

// Workspace the entry points allocate themselves comes from one stream-
// ordered pool per device that keeps its memory between calls (release
// threshold: never): mapping fresh pages for every call's workspace cost up
// to a few hundred microseconds a call.  The pool holds at most the largest
// workspace in use at once; trsm_llnn_ex and trsm_llnn_noalloc take nothing
// from it.  Without a pool (creation failed) the device's current pool.
int workspace_alloc(void **p, size_t bytes, cudaStream_t st) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static cudaMemPool_t pools[kMaxDev] = {};
    static bool tried[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    cudaMemPool_t pool = nullptr;
    if (dev >= 0 && dev < kMaxDev) {
        std::lock_guard<std::mutex> lock(mu);
        if (!tried[dev]) {
            tried[dev] = true;
            cudaMemPoolProps props{};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&pools[dev], &props) == cudaSuccess) {
                uint64_t keep = UINT64_MAX;
                cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
            } else {
                pools[dev] = nullptr;
                (void)cudaGetLastError();
            }
        }
        pool = pools[dev];
    }
    e = pool ? cudaMallocFromPoolAsync(p, bytes, pool, st) : cudaMallocAsync(p, bytes, st);
    return e == cudaSuccess ? TRSM_SUCCESS : cuda_status(e);
}

// Everything after validation.  ws: caller workspace or NULL (then it is
// allocated stream-ordered when the blocked path needs one, unless
// may_alloc is false: then TRSM_ERR_WORKSPACE).
int solve_dispatch(int dtype, int layout, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda,
                   int64_t sA, void *B, int64_t ldb, int64_t sB, int64_t batch, int64_t nb, void *ws,
                   size_t ws_bytes, bool may_alloc, cudaStream_t st, float *ms, bool tri_rhs) {
    if (ms) ms[0] = ms[1] = ms[2] = 0.f;
    if (m == 0 || n == 0 || batch == 0) return TRSM_SUCCESS;
    SmallArgs s;
    s.m = m; s.n = n; s.layout = layout;
    s.A = A; s.lda = lda; s.strideA = sA;
    s.B = B; s.ldb = ldb; s.strideB = sB;
    s.batch = batch;
    memset(s.alpha, 0, sizeof(s.alpha));
    memcpy(s.alpha, alpha, (size_t)elem_bytes(dtype));
    if (alpha_is_zero(dtype, alpha)) return launch_zero(dtype, s, st);

    if (m <= 64) {
        cudaEvent_t e0 = nullptr, e1 = nullptr;
        if (ms) {
            cudaEventCreate(&e0);
            cudaEventCreate(&e1);
            cudaEventRecord(e0, st);
        }
        int rc = launch_small(dtype, s, st);
        if (ms) {
            cudaEventRecord(e1, st);
            cudaEventSynchronize(e1);
            cudaEventElapsedTime(&ms[1], e0, e1);
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
        }
        return rc;
    }

    if (m == 128 && layout == TRSM_COL_MAJOR && n > 8 && n <= 64LL * 65535) {  // column grid: 65535 rows
        // a medium system fits on chip: the whole batch in one launch of the
        // small regime's chunked kernel instead of the blocked path system by
        // system (falls through when its alignment preconditions fail)
        cudaEvent_t e0 = nullptr, e1 = nullptr;
        if (ms) {
            cudaEventCreate(&e0);
            cudaEventCreate(&e1);
            cudaEventRecord(e0, st);
        }
        int rc = kFastNotApplicableCode;
        switch (dtype) {
            case TRSM_F32: rc = launch_fast_f32(s, st); break;
            case TRSM_F64: rc = launch_fast_f64(s, st); break;
            case TRSM_C64: rc = launch_fast_c64(s, st); break;
            default: rc = launch_fast_c128(s, st); break;
        }
        if (ms) {
            cudaEventRecord(e1, st);
            cudaEventSynchronize(e1);
            if (rc != kFastNotApplicableCode) cudaEventElapsedTime(&ms[1], e0, e1);
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
        }
        if (rc != kFastNotApplicableCode) return rc;
    }

    const int eb = elem_bytes(dtype);
    const bool nb_from_table = nb == 0;
    if (nb == 0) nb = nearest_nb(dtype, m);
    if (batch > 1 && m <= kBatchedMaxM)
        return solve_batched(dtype, layout, m, n, s.alpha, A, lda, sA, B, ldb, sB, batch, nb, ws, ws_bytes,
                             may_alloc, st);
    const size_t need = blocked_workspace_bytes((int)dtype, m, n, nb);
    // Row-major systems run through the column-major path on transposed
    // copies held after the workspace.
    const int64_t tl_bytes = layout == TRSM_ROW_MAJOR ? ((m * m * eb + 255) / 256) * 256 : 0;
    const int64_t tb_bytes = layout == TRSM_ROW_MAJOR ? ((m * n * eb + 255) / 256) * 256 : 0;
    const size_t total = need + (size_t)tl_bytes + (size_t)tb_bytes;
    void *mem = ws;
    bool owned = false;
    if (mem == nullptr || ws_bytes < total) {
        if (!may_alloc) return TRSM_ERR_WORKSPACE;
        const int ae = workspace_alloc(&mem, total, st);
        if (ae) return ae;
        owned = true;
    }
    int rc = TRSM_SUCCESS;
    for (int64_t b = 0; b < batch && rc == TRSM_SUCCESS; ++b) {
        BlockedArgs ba;
        ba.m = m; ba.n = n; ba.nb = nb;
        ba.ws = mem;
        ba.ms = ms;
        ba.tri_rhs = tri_rhs && batch == 1 && layout == TRSM_COL_MAJOR;
        ba.nb_from_table = nb_from_table;
        memcpy(ba.alpha, s.alpha, sizeof(ba.alpha));
        const char *Ab = static_cast<const char *>(A) + b * sA * eb;
        char *Bb = static_cast<char *>(B) + b * sB * eb;
        if (layout == TRSM_COL_MAJOR) {
            ba.A = Ab; ba.lda = lda;
            ba.B = Bb; ba.ldb = ldb;
            rc = blocked_solve(dtype, ba, st);
        } else {
            char *Lc = static_cast<char *>(mem) + need;
            char *Bc = Lc + tl_bytes;
            rc = launch_transpose_copy(eb, Ab, lda, Lc, m, m, m, st);
            if (!rc) rc = launch_transpose_copy(eb, Bb, ldb, Bc, m, m, n, st);
            ba.A = Lc; ba.lda = m;
            ba.B = Bc; ba.ldb = m;
            if (!rc) rc = blocked_solve(dtype, ba, st);
            // back: column-major m x n (ld m) -> row-major (ld ldb) is the
            // transpose copy of the n x m row-major view of Bc.
            if (!rc) rc = launch_transpose_copy(eb, Bc, m, Bb, ldb, n, m, st);
        }
    }
    if (owned) {
        const cudaError_t e = cudaFreeAsync(mem, st);
        if (rc == TRSM_SUCCESS && e != cudaSuccess) rc = cuda_status(e);
    }
    return rc;
}

template <typename T>
static int transpose_typed(const void *src, int64_t ld_src, void *dst, int64_t ld_dst, int64_t rows,
                           int64_t cols, cudaStream_t st, int64_t s_src, int64_t s_dst, int nz) {
    const dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32), (unsigned)nz);
    transpose_kernel<T><<<grid, dim3(32, 8), 0, st>>>(static_cast<const T *>(src), ld_src, static_cast<T *>(dst),
                                                      ld_dst, rows, cols, s_src, s_dst);
    return launch_status();
}

int launch_transpose_copy(int elem_bytes, const void *src, int64_t ld_src, void *dst, int64_t ld_dst, int64_t rows,
                          int64_t cols, cudaStream_t st, int64_t s_src, int64_t s_dst, int nz) {
    switch (elem_bytes) {
        case 4: return transpose_typed<float>(src, ld_src, dst, ld_dst, rows, cols, st, s_src, s_dst, nz);
        case 8: return transpose_typed<double>(src, ld_src, dst, ld_dst, rows, cols, st, s_src, s_dst, nz);
        default: return transpose_typed<double2>(src, ld_src, dst, ld_dst, rows, cols, st, s_src, s_dst, nz);
    }
}

// Ainv <- I (m x m, column-major, ld): CTA (x, y) writes rows x*1024 ..
// x*1024 + 1023 of columns y, y + gridDim.y, ...; a thread four rows, 256
// apart (coalesced stores, a few thousand CTAs in all).
template <typename T>
__global__ void __launch_bounds__(256) set_identity_kernel(T *__restrict__ D, int64_t m, int64_t ld) {
    const int64_t i0 = (int64_t)blockIdx.x * 1024 + threadIdx.x;
    for (int64_t j = blockIdx.y; j < m; j += gridDim.y) {
        T *col = D + j * ld;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = i0 + 256 * k;
            if (i < m) col[i] = (i == j) ? one_of<T>() : zero_of<T>();
        }
    }
}

int launch_set_identity(int dtype, void *D, int64_t m, int64_t ld, cudaStream_t st) {
    const dim3 grid((unsigned)((m + 1023) / 1024), (unsigned)(m < 512 ? m : 512));
    switch (dtype) {
        case TRSM_F32: set_identity_kernel<float><<<grid, 256, 0, st>>>(static_cast<float *>(D), m, ld); break;
        case TRSM_F64: set_identity_kernel<double><<<grid, 256, 0, st>>>(static_cast<double *>(D), m, ld); break;
        case TRSM_C64: set_identity_kernel<float2><<<grid, 256, 0, st>>>(static_cast<float2 *>(D), m, ld); break;
        default: set_identity_kernel<double2><<<grid, 256, 0, st>>>(static_cast<double2 *>(D), m, ld); break;
    }
    return launch_status();
}

}  // namespace trsm

extern "C" {

int trsm_llnn(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda, void *B,
              int64_t ldb, void *stream) {
    const int eb = elem_bytes(dtype);
    if (!eb) return -1;
    if (m < 0) return -2;
    if (n < 0) return -3;
    if (!alpha) return -4;
    if (lda < max1(m)) return -6;
    if (ldb < max1(m)) return -8;
    if (m == 0 || n == 0) return TRSM_SUCCESS;
    const bool zero = alpha_is_zero(dtype, alpha);
    if (!zero && (!A || !aligned(A, eb))) return -5;
    if (!B || !aligned(B, eb)) return -7;
    if (m <= 64 && n > 64LL * 65535) return -3;
    return solve_dispatch(dtype, TRSM_COL_MAJOR, m, n, alpha, A, lda, 0, B, ldb, 0, 1, 0, nullptr, 0, true,
                 static_cast<cudaStream_t>(stream), nullptr);
}

int trsm_llnn_strided_batched(trsm_dtype_t dtype, trsm_layout_t layout, int64_t m, int64_t n, const void *alpha,
                              const void *A, int64_t lda, int64_t strideA, void *B, int64_t ldb, int64_t strideB,
                              int64_t batch, void *stream) {
    const int eb = elem_bytes(dtype);
    if (!eb) return -1;
    if (layout != TRSM_COL_MAJOR && layout != TRSM_ROW_MAJOR) return -2;
    if (m < 0) return -3;
    if (n < 0) return -4;
    if (!alpha) return -5;
    if (lda < max1(m)) return -7;
    if (strideA < 0) return -8;
    if (ldb < (layout == TRSM_COL_MAJOR ? max1(m) : max1(n))) return -10;
    if (batch < 0) return -12;
    if (batch > 1 && strideB < (layout == TRSM_COL_MAJOR ? ldb * n : ldb * m)) return -11;
    if (m == 0 || n == 0 || batch == 0) return TRSM_SUCCESS;
    const bool zero = alpha_is_zero(dtype, alpha);
    if (!zero && (!A || !aligned(A, eb))) return -6;
    if (!B || !aligned(B, eb)) return -9;
    if (m <= 64 && n > 64LL * 65535) return -4;
    return solve_dispatch(dtype, layout, m, n, alpha, A, lda, strideA, B, ldb, strideB, batch, 0, nullptr, 0, true,
                 static_cast<cudaStream_t>(stream), nullptr);
}

int trsm_llnn_select_nb(trsm_dtype_t dtype, int64_t m, int64_t n) {
    if (!elem_bytes(dtype)) return -1;
    if (m < 0) return -2;
    if (n < 0) return -3;
    if (m <= 64) return 0;
    return nearest_nb(dtype, m);
}

size_t trsm_llnn_workspace_bytes(trsm_dtype_t dtype, int64_t m, int64_t n, int64_t nb) {
    const int eb = elem_bytes(dtype);
    if (!eb || m < 0 || n < 0) return (size_t)-1;
    if (nb != 0 && nb != 128 && nb != 256 && nb != 512) return (size_t)-1;
    if (m <= 64 || n == 0) return 0;
    if (nb == 0) nb = nearest_nb(dtype, m);
    return blocked_workspace_bytes((int)dtype, m, n, nb);
}

static int ex_common(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda,
                     void *B, int64_t ldb, int64_t nb, void *workspace, size_t ws_bytes, void *stream, float *ms) {
    const int eb = elem_bytes(dtype);
    if (!eb) return -1;
    if (m < 0) return -2;
    if (n < 0) return -3;
    if (!alpha) return -4;
    if (lda < max1(m)) return -6;
    if (ldb < max1(m)) return -8;
    if (nb != 0 && nb != 128 && nb != 256 && nb != 512) return -9;
    if (m == 0 || n == 0) {
        if (ms) ms[0] = ms[1] = ms[2] = 0.f;
        return TRSM_SUCCESS;
    }
    const bool zero = alpha_is_zero(dtype, alpha);
    if (!zero && (!A || !aligned(A, eb))) return -5;
    if (!B || !aligned(B, eb)) return -7;
    if (m <= 64 && n > 64LL * 65535) return -3;
    if (m > 64 && !zero) {
        const size_t need = blocked_workspace_bytes((int)dtype, m, n, nb ? nb : nearest_nb(dtype, m));
        if (!workspace || !aligned(workspace, 256) || ws_bytes < need) return TRSM_ERR_WORKSPACE;
    }
    return solve_dispatch(dtype, TRSM_COL_MAJOR, m, n, alpha, A, lda, 0, B, ldb, 0, 1, nb, workspace, ws_bytes, false,
                 static_cast<cudaStream_t>(stream), ms);
}

int trsm_llnn_ex(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda, void *B,
                 int64_t ldb, int64_t nb, void *workspace, size_t ws_bytes, void *stream) {
    return ex_common(dtype, m, n, alpha, A, lda, B, ldb, nb, workspace, ws_bytes, stream, nullptr);
}

int trsm_llnn_profile(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda,
                      void *B, int64_t ldb, int64_t nb, void *workspace, size_t ws_bytes, void *stream, float *ms) {
    if (!ms) return -13;
    const int rc = ex_common(dtype, m, n, alpha, A, lda, B, ldb, nb, workspace, ws_bytes, stream, ms);
    if (rc == TRSM_SUCCESS) {
        const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_status(e);
    }
    return rc;
}

int trsm_trtri_lower(trsm_dtype_t dtype, int64_t m, const void *A, int64_t lda, void *Ainv, int64_t ldinv,
                     void *stream) {
    const int eb = elem_bytes(dtype);
    if (!eb) return -1;
    if (m < 0) return -2;
    if (lda < max1(m)) return -4;
    if (ldinv < max1(m)) return -6;
    if (m == 0) return TRSM_SUCCESS;
    if (!A || !aligned(A, eb)) return -3;
    if (!Ainv || !aligned(Ainv, eb)) return -5;
    if (m > 65535) return -2;  // one grid row per column of the identity
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = launch_set_identity((int)dtype, Ainv, m, ldinv, st);
    if (rc) return rc;
    alignas(16) unsigned char one[16] = {};
    if (dtype == TRSM_F32 || dtype == TRSM_C64) {
        const float f = 1.f;
        memcpy(one, &f, sizeof f);
    } else {
        const double d = 1.0;
        memcpy(one, &d, sizeof d);
    }
    // the right-hand side is the identity: every step skips the columns that
    // are still zero (m^3/3 flops in all instead of the solve's m^3)
    return solve_dispatch(dtype, TRSM_COL_MAJOR, m, m, one, A, lda, 0, Ainv, ldinv, 0, 1, 0, nullptr, 0, true, st,
                          nullptr, /*tri_rhs=*/true);
}

int trsm_device_status(int clear) { return device_status(clear); }

int trsm_set_wait_limit(int64_t polls) { return set_first_wait_limit(polls); }

const char *trsm_status_string(int status) {
    if (status == TRSM_SUCCESS) return "success";
    if (status < 0) return "invalid argument (the negated status is its 1-based position)";
    if (status == TRSM_ERR_WORKSPACE) return "workspace missing, misaligned or too small";
    if (status == TRSM_ERR_DEVICE_TIMEOUT) return "a kernel's bounded wait on a hardware barrier expired";
    if (status >= TRSM_ERR_CUDA_BASE) return cudaGetErrorString((cudaError_t)(status - TRSM_ERR_CUDA_BASE));
    return "unknown status";
}

}  // extern "C"
