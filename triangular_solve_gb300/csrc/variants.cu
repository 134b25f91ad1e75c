// Every TRSM variant (left or right side, lower or upper triangle, A, A^T or
// A^H, unit or non-unit diagonal) through the tuned left / lower /
// non-transposed / non-unit solve.  The summary of "Hierarchical Shared
// Memory-Aware Optimization for TRSM on GPU Platforms" lists the other TRSM
// variants among its open questions; each is the same solve after a change
// of variables:
//   right side   X op(A) = alpha B  <=>  op(A)^T X^T = alpha B^T, a left-side
//                problem on B^T with the matrix op(A)^T;
//   upper        U Y = C  <=>  (J U J)(J Y) = J C with J the order reversal,
//                and J U J is lower;
//   transpose / conjugate / unit diagonal  are folded into the copy of the
//                matrix.
// So the matrix M of the left-side problem is copied, lower-triangular and
// non-unit, into a workspace (reversed when M is upper), B is reversed
// (left) or transposed (right) around the solve, and the solve itself is
// trsm_llnn.  The copies are plain elementwise kernels (O(k^2 + mn) bytes,
// not tuned); the O(k^2 n) solve carries the work.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/trsm.h"
#include "common.cuh"
#include "internal.h"

namespace trsm {

namespace {

__device__ __forceinline__ float conj_if(float v, bool) { return v; }
__device__ __forceinline__ double conj_if(double v, bool) { return v; }
__device__ __forceinline__ float2 conj_if(float2 v, bool c) { return c ? make_float2(v.x, -v.y) : v; }
__device__ __forceinline__ double2 conj_if(double2 v, bool c) { return c ? make_double2(v.x, -v.y) : v; }
template <typename T> __device__ __forceinline__ T unit_of();
template <> __device__ __forceinline__ float unit_of<float>() { return 1.f; }
template <> __device__ __forceinline__ double unit_of<double>() { return 1.0; }
template <> __device__ __forceinline__ float2 unit_of<float2>() { return make_float2(1.f, 0.f); }
template <> __device__ __forceinline__ double2 unit_of<double2>() { return make_double2(1.0, 0.0); }

// Ap (k x k, column-major, ld k), lower triangle including the diagonal:
//   Ap(i, j) = M(p, q),  (p, q) = rev ? (k-1-i, k-1-j) : (i, j),
//   M(p, q) = trans ? A(q, p) : A(p, q), conjugated when conj,
// with the diagonal set to 1 when unit (A's diagonal then never read).  Only
// the triangle of A that M's nonzero part comes from is read.
template <typename T>
__global__ void variant_matrix_kernel(const T *__restrict__ A, int64_t lda, int64_t k, T *__restrict__ Ap,
                                      bool trans, bool rev, bool conj, bool unit) {
    const int64_t j = blockIdx.y;
    for (int64_t i = j + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < k; i += (int64_t)gridDim.x * blockDim.x) {
        T v;
        if (unit && i == j) {
            v = unit_of<T>();
        } else {
            const int64_t p = rev ? k - 1 - i : i, q = rev ? k - 1 - j : j;
            const int64_t r = trans ? q : p, c = trans ? p : q;
            v = conj_if(A[c * lda + r], conj);
        }
        Ap[j * k + i] = v;
    }
}

// Reverse the order of the rows of a rows x cols column-major matrix.
template <typename T>
__global__ void reverse_rows_kernel(T *__restrict__ B, int64_t ld, int64_t rows) {
    const int64_t j = blockIdx.y;
    T *col = B + j * ld;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows / 2; i += (int64_t)gridDim.x * blockDim.x) {
        const T a = col[i], b = col[rows - 1 - i];
        col[i] = b;
        col[rows - 1 - i] = a;
    }
}

unsigned grid_x(int64_t work) { return (unsigned)((work + 255) / 256 < 64 ? (work + 255) / 256 : 64); }

template <typename T>
int matrix_copy(const void *A, int64_t lda, int64_t k, void *Ap, bool trans, bool rev, bool conj, bool unit,
                cudaStream_t st) {
    variant_matrix_kernel<T><<<dim3(grid_x(k), (unsigned)k), 256, 0, st>>>(static_cast<const T *>(A), lda, k,
                                                                           static_cast<T *>(Ap), trans, rev,
                                                                           conj, unit);
    return launch_status();
}

template <typename T>
int reverse_rows(void *B, int64_t ld, int64_t rows, int64_t cols, cudaStream_t st) {
    if (rows < 2 || cols == 0) return TRSM_SUCCESS;
    reverse_rows_kernel<T><<<dim3(grid_x(rows / 2), (unsigned)cols), 256, 0, st>>>(static_cast<T *>(B), ld, rows);
    return launch_status();
}

template <typename T>
int variant_solve(trsm_dtype_t dtype, bool right, bool trans, bool rev, bool conj, bool unit, int64_t m, int64_t n,
                  const void *alpha, const void *A, int64_t lda, void *B, int64_t ldb, cudaStream_t st) {
    const int64_t k = right ? n : m, other = right ? m : n;
    const size_t a_bytes = round256(k * k * (int64_t)sizeof(T));
    const size_t b_bytes = right ? (size_t)round256(n * m * (int64_t)sizeof(T)) : 0;
    void *ws = nullptr;
    const int ae = workspace_alloc(&ws, a_bytes + b_bytes, st);
    if (ae) return ae;
    cudaError_t e = cudaSuccess;
    void *Ap = ws;
    void *Bp = right ? static_cast<char *>(ws) + a_bytes : B;
    const int64_t ldp = right ? n : ldb;
    int rc = matrix_copy<T>(A, lda, k, Ap, trans, rev, conj, unit, st);
    if (!rc && right) rc = launch_transpose_copy((int)sizeof(T), B, ldb, Bp, n, n, m, st);  // B^T
    if (!rc && rev) rc = reverse_rows<T>(Bp, ldp, k, other, st);
    if (!rc) rc = trsm_llnn(dtype, k, other, alpha, Ap, k, Bp, ldp, st);
    if (!rc && rev) rc = reverse_rows<T>(Bp, ldp, k, other, st);
    if (!rc && right) rc = launch_transpose_copy((int)sizeof(T), Bp, n, B, ldb, m, n, st);
    e = cudaFreeAsync(ws, st);
    if (!rc && e != cudaSuccess) rc = cuda_status(e);
    return rc;
}

}  // namespace

}  // namespace trsm

extern "C" int trsm_general(trsm_dtype_t dtype, trsm_side_t side, trsm_uplo_t uplo, trsm_op_t trans,
                            trsm_diag_t diag, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda,
                            void *B, int64_t ldb, void *stream) {
    using namespace trsm;
    const int eb = dtype == TRSM_F32 ? 4 : dtype == TRSM_F64 || dtype == TRSM_C64 ? 8 : dtype == TRSM_C128 ? 16 : 0;
    if (!eb) return -1;
    if (side != TRSM_LEFT && side != TRSM_RIGHT) return -2;
    if (uplo != TRSM_LOWER && uplo != TRSM_UPPER) return -3;
    if (trans != TRSM_NOTRANS && trans != TRSM_TRANS && trans != TRSM_CONJTRANS) return -4;
    if (diag != TRSM_NONUNIT && diag != TRSM_UNIT) return -5;
    if (m < 0) return -6;
    if (n < 0) return -7;
    if (!alpha) return -8;
    const int64_t k = side == TRSM_LEFT ? m : n;
    if (lda < (k > 1 ? k : 1)) return -10;
    if (ldb < (m > 1 ? m : 1)) return -12;
    if (m == 0 || n == 0) return TRSM_SUCCESS;
    if (!B || reinterpret_cast<uintptr_t>(B) % eb) return -11;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool cplx = dtype == TRSM_C64 || dtype == TRSM_C128;
    bool zero = true;
    for (int i = 0; i < (cplx ? 2 : 1); ++i) {
        if (eb == 4 || dtype == TRSM_C64) zero = zero && static_cast<const float *>(alpha)[i] == 0.f;
        else zero = zero && static_cast<const double *>(alpha)[i] == 0.0;
    }
    if (zero) return trsm_llnn(dtype, m, n, alpha, nullptr, m > 1 ? m : 1, B, ldb, stream);  // B <- 0, A unread
    if (!A || reinterpret_cast<uintptr_t>(A) % eb) return -9;
    if (side == TRSM_LEFT && uplo == TRSM_LOWER && trans == TRSM_NOTRANS && diag == TRSM_NONUNIT)
        return trsm_llnn(dtype, m, n, alpha, A, lda, B, ldb, stream);
    if (k > 65535 || (side == TRSM_LEFT ? n : m) > 65535) return side == TRSM_LEFT ? -7 : -6;  // copy grids
    // the left-side problem's matrix: op(A) (left) or op(A)^T (right)
    const bool right = side == TRSM_RIGHT;
    const bool tr = right ? trans == TRSM_NOTRANS : trans != TRSM_NOTRANS;
    const bool conj = cplx && trans == TRSM_CONJTRANS;
    const bool lower = (uplo == TRSM_LOWER) != tr;  // that matrix is lower triangular
    const bool unit = diag == TRSM_UNIT;
    switch (dtype) {
        case TRSM_F32: return variant_solve<float>(dtype, right, tr, !lower, conj, unit, m, n, alpha, A, lda, B, ldb, st);
        case TRSM_F64: return variant_solve<double>(dtype, right, tr, !lower, conj, unit, m, n, alpha, A, lda, B, ldb, st);
        case TRSM_C64: return variant_solve<float2>(dtype, right, tr, !lower, conj, unit, m, n, alpha, A, lda, B, ldb, st);
        default: return variant_solve<double2>(dtype, right, tr, !lower, conj, unit, m, n, alpha, A, lda, B, ldb, st);
    }
}
