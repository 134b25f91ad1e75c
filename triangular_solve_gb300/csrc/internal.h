// Internal interfaces between the C ABI (api.cu) and the kernel launchers.
#pragma once

#include <cuda.h>

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

namespace trsm {

// One (strided-batched) solve, arguments already validated.  alpha holds one
// value of the element type (up to two doubles).
struct SmallArgs {
    int64_t m, n;
    int layout;  // 0 column-major, 1 row-major
    const void *A;
    int64_t lda, strideA;
    void *B;
    int64_t ldb, strideB;
    int64_t batch;
    alignas(16) unsigned char alpha[16];
};

// Small regime, m <= 64: one launch over the whole batch.  colreg: one
// thread per RHS column (n > 8); rowlane: one warp per system (n <= 8).
int launch_colreg_f32(const SmallArgs &a, cudaStream_t st);
int launch_colreg_f64(const SmallArgs &a, cudaStream_t st);
int launch_colreg_c64(const SmallArgs &a, cudaStream_t st);
int launch_colreg_c128(const SmallArgs &a, cudaStream_t st);
int launch_rowlane_f32(const SmallArgs &a, cudaStream_t st);
int launch_rowlane_f64(const SmallArgs &a, cudaStream_t st);
int launch_rowlane_c64(const SmallArgs &a, cudaStream_t st);
int launch_rowlane_c128(const SmallArgs &a, cudaStream_t st);
// m <= 8: one thread per (system, right-hand-side column).
int launch_tiny_f32(const SmallArgs &a, cudaStream_t st);
int launch_tiny_f64(const SmallArgs &a, cudaStream_t st);
int launch_tiny_c64(const SmallArgs &a, cudaStream_t st);
int launch_tiny_c128(const SmallArgs &a, cudaStream_t st);

// Fast path of the thread-per-column kernel for aligned full-size systems
// (m in {8, 16, 32, 48, 64}, and 128 for batches of medium systems); returns
// kFastNotApplicable (-100000) when its preconditions do not hold.
int launch_fast_f32(const SmallArgs &a, cudaStream_t st);
int launch_fast_f64(const SmallArgs &a, cudaStream_t st);
int launch_fast_c64(const SmallArgs &a, cudaStream_t st);
int launch_fast_c128(const SmallArgs &a, cudaStream_t st);

// alpha == 0: B <- 0 without reading A.
int launch_zero_f32(const SmallArgs &a, cudaStream_t st);
int launch_zero_f64(const SmallArgs &a, cudaStream_t st);
int launch_zero_c64(const SmallArgs &a, cudaStream_t st);
int launch_zero_c128(const SmallArgs &a, cudaStream_t st);

// Blocked path for one column-major system, m > 64.
struct BlockedArgs {
    int64_t m, n, nb;
    const void *A;
    int64_t lda;
    void *B;
    int64_t ldb;
    alignas(16) unsigned char alpha[16];
    void *ws;        // >= blocked_workspace_bytes(elem, m, n, nb), 256-byte aligned
    float *ms;       // optional: per-phase milliseconds (profiling entry)
    // B holds the identity (alpha = 1): block row t's solve and update touch
    // only its first (t+1) nb columns (the triangular inverse)
    bool tri_rhs = false;
    // nb is the table's choice (the caller passed 0), so a path with its own
    // block size (few right-hand sides: 128) may take over
    bool nb_from_table = true;
};

// Bytes of workspace the blocked path needs: the inverted diagonal blocks
// (ceil(m/nb) x nb x nb), then two nb x panel_ld(n) row-major panels (X_t,
// and the transposed block row R_t the single-precision apply reads), each
// rounded up to 256 bytes.
inline int64_t panel_ld(int64_t n) { return ((n > 0 ? n : 1) + 3) / 4 * 4; }
inline int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }
// f32 adds the TF32 head/tail panels of the tensor-core products
// (tc_panel_bytes: the A operand -- L panel or D_t^-1 --, the X operand and
// the split X_t the apply leaves for the update, two copies each, K-major;
// or, when the look-ahead form applies and needs more, its panels:
// tc_fused_bytes).
// c64 adds the real-form operands of its tensor-core products
// (tc_panel_bytes_c64: A' = m x 2nb, X' = 2n x 2nb and the split X_t' the
// apply leaves for the update, two copies each; or the look-ahead panels,
// tc_fused_bytes_c64, when that form applies and needs more).
size_t tc_panel_bytes(int64_t m, int64_t n, int64_t nb);
size_t tc_panel_bytes_c64(int64_t m, int64_t n, int64_t nb);
// The few-right-hand-sides path (n <= kFewMaxN, few_rhs.cuh) keeps its own
// data in the same workspace: the inverted diagonal blocks of kFewNb rows,
// then the published copy of X (block row by block row, column by column).
constexpr int64_t kFewNb = 128;
constexpr int kFewMaxN = 8;
inline size_t few_rhs_bytes(int elem_bytes, int64_t m, int64_t n) {
    const int64_t tb = (m + kFewNb - 1) / kFewNb;
    return (size_t)(round256(tb * kFewNb * kFewNb * elem_bytes) + round256(tb * n * kFewNb * elem_bytes));
}
inline size_t blocked_workspace_bytes(int dtype, int64_t m, int64_t n, int64_t nb) {
    const int elem_bytes = dtype == 0 ? 4 : dtype == 3 ? 16 : 8;
    const int64_t tb = (m + nb - 1) / nb;
    size_t b = (size_t)(round256(tb * nb * nb * elem_bytes) + 2 * round256(nb * panel_ld(n) * elem_bytes));
    if (dtype == 0) b += tc_panel_bytes(m, n, nb);
    if (dtype == 2) b += tc_panel_bytes_c64(m, n, nb);
    if (n <= kFewMaxN) {
        const size_t f = few_rhs_bytes(elem_bytes, m, n);
        if (f > b) b = f;
    }
    return b;
}

// Tensor-core (tcgen05, 3xTF32) f32 products of the blocked path; see
// tc_gemm.cuh / tc_gemm.cu.  tc_update_f32 with X == nullptr takes the split
// X_t that tc_apply_f32(..., emit_split = true) left in the panels.
bool tc_update_usable(int64_t M, int64_t N, int64_t K);
bool tc_apply_usable(int64_t mb, int64_t N);
int tc_update_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *X, int64_t ldx,
                  float *C, int64_t ldc, float beta, int64_t Mmax, void *panels, cudaStream_t st);
bool tc_apply_usable_c64(int64_t mb, int64_t N);
int tc_apply_c64(int64_t mb, int64_t N, const float2 *Wt, int64_t nb, float2 *Bt, int64_t ldb, float2 gamma,
                 int64_t Mmax, void *panels, bool emit_split, cudaStream_t st);
int tc_update_c64(int64_t M, int64_t N, int64_t K, const float2 *A, int64_t lda, const float2 *X, int64_t ldx,
                  float2 *C, int64_t ldc, float2 beta, int64_t Mmax, void *panels, cudaStream_t st);
int tc_apply_f32(int64_t mb, int64_t N, const float *Wt, int64_t nb, float *Bt, int64_t ldb, float gamma,
                 int64_t Mmax, void *panels, bool emit_split, cudaStream_t st);
// Look-ahead form of the f32 solve on the tensor cores (tc_gemm.cu): after
// the inversion, tc_fused_prepare once, then tc_fused_step for t = 0 .. tb-1.
bool tc_fused_usable(int64_t m, int64_t n, int64_t nb);
size_t tc_fused_bytes(int64_t m, int64_t n, int64_t nb);
int tc_fused_prepare(int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W, const float *B,
                     int64_t ldb, void *panels, cudaStream_t st, bool tri = false);
int tc_fused_step(int64_t t, int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W,
                  float *B, int64_t ldb, float alpha, void *panels, cudaStream_t st, bool tri = false);
// The same for c64, in real form with interleaved K (tc_gemm.cu).
bool tc_fused_usable_c64(int64_t m, int64_t n, int64_t nb);
size_t tc_fused_bytes_c64(int64_t m, int64_t n, int64_t nb);
int tc_fused_prepare_c64(int64_t m, int64_t n, int64_t nb, const float2 *L, int64_t lda, const float2 *W,
                         const float2 *B, int64_t ldb, void *panels, cudaStream_t st, bool tri = false);
int tc_fused_step_c64(int64_t t, int64_t m, int64_t n, int64_t nb, const float2 *L, int64_t lda, const float2 *W,
                      float2 *B, int64_t ldb, float2 alpha, void *panels, cudaStream_t st, bool tri = false);
// Tiled TMA tensor map of an f32 tensor (see tc_gemm.cu).
int encode_f32_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                   const uint32_t *box, bool swizzle128);
// Device status word of the bounded waits: its device address (for the
// kernels), and its value (synchronises the device).
int device_status_word(int **out);
int device_status(int clear);
// Polls of the first bounded wait on each item of the batched f32 small
// kernel: the compiled limit unless trsm_set_wait_limit lowered it.
uint32_t first_wait_limit();
int set_first_wait_limit(int64_t polls);

// Blocked path over a strided batch of column-major systems, one launch
// sequence for all of them (blocked_launch.cuh); batch <= 65535 (the grid's
// system dimension), strideA = 0 for one A shared by every system.
struct BatchedBlockedArgs {
    int64_t m, n, nb;
    const void *A;
    int64_t lda, strideA;
    void *B;
    int64_t ldb, strideB;
    int64_t batch;
    alignas(16) unsigned char alpha[16];
    void *ws;  // >= batched_workspace_bytes(...), 256-byte aligned
};
inline size_t batched_workspace_bytes(int dtype, int64_t m, int64_t n, int64_t nb, int64_t batch, bool shared_a) {
    const int64_t eb = dtype == 0 ? 4 : dtype == 3 ? 16 : 8;
    const int64_t tb = (m + nb - 1) / nb;
    return (size_t)(round256((shared_a ? 1 : batch) * tb * nb * nb * eb) + 2 * round256(batch * nb * panel_ld(n) * eb));
}
int blocked_solve_batched_f32(const BatchedBlockedArgs &a, cudaStream_t st);
int blocked_solve_batched_f64(const BatchedBlockedArgs &a, cudaStream_t st);
int blocked_solve_batched_c64(const BatchedBlockedArgs &a, cudaStream_t st);
int blocked_solve_batched_c128(const BatchedBlockedArgs &a, cudaStream_t st);

int blocked_solve_f32(const BlockedArgs &a, cudaStream_t st);
int blocked_solve_f64(const BlockedArgs &a, cudaStream_t st);
int blocked_solve_c64(const BlockedArgs &a, cudaStream_t st);
int blocked_solve_c128(const BlockedArgs &a, cudaStream_t st);

// The dispatch behind every solve entry point, after argument checks: alpha
// = 0, the small regime (m <= 64), batches of m = 128 systems, the blocked
// path.  ws / ws_bytes: the blocked path's workspace (plus the transposed
// copies of row-major systems); when it is missing or too small the call
// allocates one with cudaMallocAsync on st if may_alloc, else returns
// TRSM_ERR_WORKSPACE before launching anything.  nb = 0: the table's block
// size.  ms: optional phase times (synchronises st).
int solve_dispatch(int dtype, int layout, int64_t m, int64_t n, const void *alpha, const void *A, int64_t lda,
                   int64_t sA, void *B, int64_t ldb, int64_t sB, int64_t batch, int64_t nb, void *ws,
                   size_t ws_bytes, bool may_alloc, cudaStream_t st, float *ms, bool tri_rhs = false);

// Row-major <-> column-major copy of a rows x cols matrix (out-of-place),
// used to run row-major inputs through the column-major blocked path.
// With nz > 1: nz such copies, src and dst advancing by s_src / s_dst elements.
// Workspace of the entry points that allocate their own: the library's
// per-device stream-ordered pool (api.cu); freed with cudaFreeAsync.
int workspace_alloc(void **p, size_t bytes, cudaStream_t st);
int launch_transpose_copy(int elem_bytes, const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                          int64_t rows, int64_t cols, cudaStream_t st, int64_t s_src = 0, int64_t s_dst = 0,
                          int nz = 1);

}  // namespace trsm
