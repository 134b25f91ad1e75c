/*
 * trsm.h -- C ABI of the GB300 (sm_103a) triangular-solve library
 *           (libtrsm_gb300.so).
 *
 * One operation, in four element types:
 *
 *     solve  L * X = alpha * B  for X, overwriting B,
 *
 * where L is the lower triangle (diagonal included) of the square matrix A.
 * The strictly upper triangle of A is never read.  The diagonal is not
 * assumed to be one.  This is the left-side, lower-triangular,
 * non-transposed, non-unit-diagonal TRSM studied in "Hierarchical Shared
 * Memory-Aware Optimization for TRSM on GPU Platforms" (developinglight.com
 * summary, opening paragraph and "One framework, several paths"), and the
 * SOLVE_TRI operation of llama.cpp PR 17457 ("SOLVE_TRI CUDA kernel for small
 * matrices"), which adds batching over independent systems.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - A and B are DEVICE pointers owned by the caller.  A is only read; B is
 *    overwritten with X.  Element types: TRSM_F32 float, TRSM_F64 double,
 *    TRSM_C64 interleaved {float re, im}, TRSM_C128 interleaved
 *    {double re, im}.  A and B must be aligned to their element size.
 *  - alpha is a HOST pointer to one value of the element type (one float,
 *    one double, or two floats / two doubles for the complex types).
 *  - Leading dimensions and batch strides count ELEMENTS, not bytes (the
 *    reviewers of llama.cpp PR 17457 asked for strides in units of the
 *    element type).  Column-major: element (i, j) sits at j*ld + i and
 *    ld >= max(1, rows).  Row-major: at i*ld + j and ld >= max(1, cols).
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call is asynchronous and stream-ordered: it enqueues
 *    kernels and returns; there is no host synchronisation inside.
 *  - Quick returns: m == 0, n == 0 or batch == 0 returns TRSM_SUCCESS without
 *    touching memory.  alpha == 0 sets B to zero without reading A (BLAS).
 *  - A zero (or non-finite) diagonal entry is not an error: IEEE inf/NaN
 *    propagate into X and the call still returns TRSM_SUCCESS (llama.cpp PR
 *    17457 removed its division-by-zero guard because a zero pivot means the
 *    data is already corrupt).
 *  - Argument errors return a negative status -k, k the 1-based position of
 *    the first invalid argument (LAPACK xerbla style), and launch nothing.
 *    A CUDA error returns TRSM_ERR_CUDA_BASE + cudaError_t.
 *  - Work runs entirely in this library's kernels on the current device;
 *    there is no CPU fallback.
 */
#ifndef TRSM_GB300_H
#define TRSM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TRSM_F32 = 0, TRSM_F64 = 1, TRSM_C64 = 2, TRSM_C128 = 3 } trsm_dtype_t;
typedef enum { TRSM_COL_MAJOR = 0, TRSM_ROW_MAJOR = 1 } trsm_layout_t;
/* the other TRSM variants (trsm_general) */
typedef enum { TRSM_LEFT = 0, TRSM_RIGHT = 1 } trsm_side_t;
typedef enum { TRSM_LOWER = 0, TRSM_UPPER = 1 } trsm_uplo_t;
typedef enum { TRSM_NOTRANS = 0, TRSM_TRANS = 1, TRSM_CONJTRANS = 2 } trsm_op_t;
typedef enum { TRSM_NONUNIT = 0, TRSM_UNIT = 1 } trsm_diag_t;

#define TRSM_SUCCESS 0
#define TRSM_ERR_WORKSPACE 900      /* caller workspace too small or misaligned */
#define TRSM_ERR_DEVICE_TIMEOUT 901 /* a kernel's bounded wait expired (see trsm_device_status) */
#define TRSM_ERR_CUDA_BASE 1000     /* TRSM_ERR_CUDA_BASE + cudaError_t */

/*
 * Single column-major system:  L X = alpha B,  A is m x m (lda >= max(1,m)),
 * B is m x n (ldb >= max(1,m)).
 *
 * m <= 64 runs the small-regime shared-memory kernel (one launch).  Larger m
 * runs the blocked path of "Hierarchical Shared Memory-Aware Optimization for
 * TRSM on GPU Platforms" (diagonal-block inversion, then per block row an
 * apply X_t = D_t^{-1} R_t and a trailing GEMM update), with the block size
 * NB taken from the library's compile-time table; with n <= 8 right-hand
 * sides, m > 512 and 16-byte aligned columns of A, the same algorithm runs
 * as one cooperative persistent launch over 128-row block rows (also through
 * trsm_llnn_ex when its nb is 0 or 128).  The blocked path needs a
 * device workspace of trsm_llnn_workspace_bytes(dtype, m, n, 0) bytes; this
 * entry point takes it, ordered on `stream`, from a memory pool the library
 * keeps per device (cudaMallocFromPoolAsync / cudaFreeAsync; the pool keeps
 * its memory between calls, up to the largest workspace in use at once).
 * Use trsm_llnn_ex to pass your own, trsm_llnn_noalloc to allocate nothing.
 *
 * Arguments: 1 dtype, 2 m, 3 n, 4 alpha, 5 A, 6 lda, 7 B, 8 ldb, 9 stream.
 */
int trsm_llnn(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha,
              const void *A, int64_t lda, void *B, int64_t ldb, void *stream);

/*
 * `batch` independent systems; system b's A starts at A + b*strideA and its
 * B at B + b*strideB (element strides; any value, including 0 for a shared
 * A, is accepted for A; strideB must keep the B matrices disjoint).
 * `layout` applies to both A and B.  This is the batched SOLVE_TRI of
 * llama.cpp PR 17457 (its 4-D tensors flattened to one batch index).
 *
 * m <= 64: one launch of the small-regime kernel over the whole batch.
 * m = 128 (column-major, 16-byte aligned columns): one launch of the
 * chunked on-chip kernel over the whole batch.  Other m <= 2048: the blocked
 * path over the whole batch in one sequence of launches (the system index in
 * every kernel's grid; one inversion for all systems when strideA == 0),
 * chunked to at most 65535 systems and 1 GiB of workspace per chunk.
 * Larger m: the blocked path system by system.  The workspace of the blocked
 * paths comes from the library's pool, ordered on `stream`, as in trsm_llnn.
 *
 * Arguments: 1 dtype, 2 layout, 3 m, 4 n, 5 alpha, 6 A, 7 lda, 8 strideA,
 * 9 B, 10 ldb, 11 strideB, 12 batch, 13 stream.
 */
int trsm_llnn_strided_batched(trsm_dtype_t dtype, trsm_layout_t layout, int64_t m, int64_t n,
                              const void *alpha, const void *A, int64_t lda, int64_t strideA,
                              void *B, int64_t ldb, int64_t strideB, int64_t batch,
                              void *stream);

/*
 * trsm_llnn_strided_batched on HOST buffers: A and B are host pointers (page-
 * locked memory lets the copies run asynchronously and overlap; pageable
 * memory works but serialises them), same arguments, layouts, strides and
 * validation as trsm_llnn_strided_batched.  B is overwritten with X.
 * The pages describe no such entry point; it exists for callers whose data
 * lives in host memory.
 *
 * The batch is cut into up to eight chunks that flow through a three-stage
 * pipeline -- host-to-device copy, solve, device-to-host copy -- on three
 * internal streams, so the copy in of one chunk, the solve of the previous
 * one and the copy out of the one before run at the same time.  The internal
 * streams are forked from `stream` and joined back to it with events.  They
 * and a ring of three device buffer sets are kept per (device, caller
 * stream) for the life of the process: the first call on a stream creates
 * the streams and allocates the buffers with cudaMalloc; the buffers only
 * grow, so later calls of the same or smaller size allocate nothing.  A call
 * that needs larger buffers frees the old ones with cudaFree first, which
 * waits for the whole device (a synchronising grow).  The call is
 * stream-ordered like the others: it returns once the work is enqueued, and
 * X is in B only when `stream` has reached the end of this call's work
 * (synchronise it before reading B).  A and B must stay valid and B must not
 * be read or written by the host until then.  Returns the first error of the
 * copies or solves (TRSM_ERR_CUDA_BASE + cudaError_t, or the solve's status).
 */
int trsm_llnn_strided_batched_host(trsm_dtype_t dtype, trsm_layout_t layout, int64_t m, int64_t n,
                                   const void *alpha, const void *A, int64_t lda, int64_t strideA,
                                   void *B, int64_t ldb, int64_t strideB, int64_t batch, void *stream);

/*
 * Block size NB the blocked path uses for (dtype, m, n): the entry of the
 * compile-time "size x type -> block size" table of the nearest tabulated m
 * ("Hierarchical Shared Memory-Aware Optimization for TRSM on GPU
 * Platforms", adaptive blocking: offline sweep, online nearest-match lookup).
 * Returns 0 when m <= 64 (no blocking) and a negative status for invalid
 * arguments (1 dtype, 2 m, 3 n).
 */
int trsm_llnn_select_nb(trsm_dtype_t dtype, int64_t m, int64_t n);

/*
 * Device workspace in bytes the blocked path needs for (dtype, m, n) with
 * block size nb (nb == 0: the table's choice; otherwise one of 128, 256,
 * 512).  0 when m <= 64.  Returns (size_t)-1 for invalid arguments.
 * The workspace holds the inverted diagonal blocks D_t^{-1} (m x NB) and one
 * NB x n panel of X; with n <= 8 it is at least what the few-right-hand-side
 * kernel keeps there (the inverted 128-row diagonal blocks and a copy of X,
 * each rounded up to 256 bytes).
 */
size_t trsm_llnn_workspace_bytes(trsm_dtype_t dtype, int64_t m, int64_t n, int64_t nb);

/*
 * trsm_llnn with an explicit block size and a caller-owned workspace.
 * nb: 0 = table choice, else 128, 256 or 512 (ignored when m <= 64).
 * workspace: device pointer, 256-byte aligned, at least
 * trsm_llnn_workspace_bytes(dtype, m, n, nb) bytes (may be NULL when that is
 * 0).  The call allocates nothing.  The workspace must not be used by
 * another call until this call's work on `stream` has finished.
 * Returns TRSM_ERR_WORKSPACE when the workspace is too small or misaligned.
 *
 * Arguments: 1 dtype, 2 m, 3 n, 4 alpha, 5 A, 6 lda, 7 B, 8 ldb, 9 nb,
 * 10 workspace, 11 ws_bytes, 12 stream.
 */
int trsm_llnn_ex(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha,
                 const void *A, int64_t lda, void *B, int64_t ldb, int64_t nb,
                 void *workspace, size_t ws_bytes, void *stream);

/*
 * trsm_llnn_ex, additionally timing its phases with CUDA events on `stream`
 * and SYNCHRONISING the stream before returning (a profiling entry, not for
 * production use):  ms[0] diagonal-block inversion, ms[1] the block applies
 * X_t = D_t^{-1} R_t, ms[2] the trailing GEMM updates, in milliseconds (the
 * split reported in "Hierarchical Shared Memory-Aware Optimization for TRSM
 * on GPU Platforms", Table 3).  For m <= 64 the whole solve is reported in
 * ms[1] and the other two are 0; for the few-right-hand-sides launch the
 * applies and updates run together and are reported in ms[2] (ms[1] = 0).
 * ms must point to 3 host floats.
 *
 * Arguments: 1..12 as trsm_llnn_ex, 13 ms.
 */
int trsm_llnn_profile(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha,
                      const void *A, int64_t lda, void *B, int64_t ldb, int64_t nb,
                      void *workspace, size_t ws_bytes, void *stream, float *ms);

/*
 * Every TRSM variant, with the BLAS xTRSM meaning ("Hierarchical Shared
 * Memory-Aware Optimization for TRSM on GPU Platforms" leaves the variants
 * beyond the left / lower / no-transpose case open):
 *   side TRSM_LEFT:   op(A) X = alpha B,  A is m x m (lda >= max(1,m))
 *   side TRSM_RIGHT:  X op(A) = alpha B,  A is n x n (lda >= max(1,n))
 * with op(A) = A, A^T or A^H (TRSM_CONJTRANS; the same as A^T for real
 * types), only the triangle `uplo` of A read, and for TRSM_UNIT the diagonal
 * taken as 1 and never read.  B is m x n, column-major (ldb >= max(1,m)), and
 * is overwritten with X.
 *
 * The left / lower / no-transpose / non-unit case is trsm_llnn itself.  Any
 * other is mapped onto it: the matrix of the equivalent left-side lower
 * problem (op(A), or op(A)^T for the right side, reversed in row and column
 * order when it is upper, with the unit diagonal written in) is copied into
 * a workspace from the library's pool, ordered on `stream` (k^2 elements,
 * plus m n for the right side), B is reversed in row order or
 * transposed into the workspace around the solve, and trsm_llnn runs on it.
 * alpha = 0 sets B to zero without reading A.  The order of A and the other
 * dimension are limited to 65535 for the variants that copy.
 *
 * Arguments: 1 dtype, 2 side, 3 uplo, 4 trans, 5 diag, 6 m, 7 n, 8 alpha,
 * 9 A, 10 lda, 11 B, 12 ldb, 13 stream.
 */
int trsm_general(trsm_dtype_t dtype, trsm_side_t side, trsm_uplo_t uplo, trsm_op_t trans,
                 trsm_diag_t diag, int64_t m, int64_t n, const void *alpha,
                 const void *A, int64_t lda, void *B, int64_t ldb, void *stream);

/*
 * Triangular inverse (TRTRI, lower, non-unit):  Ainv = L^{-1}, the inverse
 * of the lower triangle of A (m x m, lda >= max(1,m); the strictly upper part
 * of A is never read), into Ainv (m x m, column-major, ldinv >= max(1,m)),
 * whose strictly upper part is set to zero.  Computed as the solve
 * L Ainv = I on `stream` (Ainv is set to the identity, then solved in place
 * by the path trsm_llnn takes, with the same workspace allocation).  Every
 * product of that solve is restricted to the columns of the identity that
 * can be nonzero at its step, so the inverse costs TRTRI's m^3/3 flops
 * rather than the m^3 of a general solve; the diagonal-block inverses of
 * "Hierarchical Shared Memory-Aware Optimization for TRSM on GPU Platforms"
 * are its first phase.  Ainv must not overlap A.
 * A zero on the diagonal gives IEEE infinities / NaN, no status.
 *
 * Arguments: 1 dtype, 2 m, 3 A, 4 lda, 5 Ainv, 6 ldinv, 7 stream.
 */
int trsm_trtri_lower(trsm_dtype_t dtype, int64_t m, const void *A, int64_t lda,
                     void *Ainv, int64_t ldinv, void *stream);

/*
 * Size in bytes of the device array trsm_llnn_noalloc uses as its workspace
 * (32 MiB; every GPU that loads the library holds it until the process
 * exits).
 */
#define TRSM_NOALLOC_SCRATCH_BYTES (32 * 1024 * 1024)

/*
 * trsm_llnn for callers that cannot allocate device memory -- for example a
 * library embedded in a host application that owns all device memory
 * through its own pool, or a latency-sensitive path on which cudaMalloc and
 * cudaFree (which may synchronise the device) are not acceptable.  The
 * pages describe no such entry point; it has no counterpart there.
 *
 * Same operation, arguments and validation as trsm_llnn (1 dtype, 2 m, 3 n,
 * 4 alpha, 5 A, 6 lda, 7 B, 8 ldb, 9 stream; column-major, one system), but
 * the call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  m <= 64 needs no workspace.  For m > 64 the blocked path's
 * workspace lives in a fixed device array of TRSM_NOALLOC_SCRATCH_BYTES
 * inside the library.  The block size is trsm_llnn's (the table's) when its
 * workspace (trsm_llnn_workspace_bytes(dtype, m, n, 0)) fits the array,
 * else the largest smaller one (256, 128) whose workspace fits -- the same
 * solve with narrower blocks, so results agree with trsm_llnn to rounding;
 * a problem that fits at none is rejected with TRSM_ERR_WORKSPACE before
 * anything is launched.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  All calls on a device share the
 * array and it keeps the last call's contents (nothing in it needs to start
 * at zero), so calls whose GPU work overlaps -- unordered streams, or
 * several host threads -- race on it and must be serialised by the caller.
 */
int trsm_llnn_noalloc(trsm_dtype_t dtype, int64_t m, int64_t n, const void *alpha,
                      const void *A, int64_t lda, void *B, int64_t ldb, void *stream);

/*
 * Device-side status of the current device: the kernels that wait on
 * hardware barriers (the tensor-core update of the f32 blocked path) bound
 * every wait; when one expires the kernel abandons its tile and records
 * TRSM_ERR_DEVICE_TIMEOUT here instead of hanging.  Synchronises the current
 * device, returns TRSM_SUCCESS or TRSM_ERR_DEVICE_TIMEOUT (or a CUDA error
 * status), and resets the word to TRSM_SUCCESS when `clear` is non-zero.
 * No counterpart on the pages.
 */
int trsm_device_status(int clear);

/*
 * Testing hook for the bounded waits: sets how many times the batched f32
 * small-regime kernel (the one that streams systems through the TMA engine)
 * polls for each item's copies before it gives up, records
 * TRSM_ERR_DEVICE_TIMEOUT (see trsm_device_status), lets the copies already
 * in flight land (those waits keep the full limit), and returns with the
 * item unsolved.  polls = 0 makes every such wait expire at once, so a test
 * can exercise the timeout path without a fault or a hang; a negative value
 * restores the compiled limit.  Applies to launches made after the call, on
 * every device.  Not for production use.  No counterpart on the pages.
 */
int trsm_set_wait_limit(int64_t polls);

/* Static, human-readable text for a status code returned by this library. */
const char *trsm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* TRSM_GB300_H */
