// Host side of the tensor-core f32 trailing update: TF32 head/tail split of
// the two panels, tensor maps for the TMA loads, launch, and the device
// status word that the kernels' bounded waits report to.
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_gemm.cuh"
#include "tc_side.h"

namespace trsm {

namespace {

static __device__ int g_device_status;  // TRSM_ERR_DEVICE_TIMEOUT when a bounded wait expired

constexpr int kMaxDev = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDev] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int encoder(PFN_cuTensorMapEncodeTiled_v12000 *out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_status(e);
        if (q != cudaDriverEntryPointSuccess || !fn) return TRSM_ERR_CUDA_BASE + (int)cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return TRSM_SUCCESS;
}

// K-major rows x k matrix (row stride ld floats), box 32 (k) x box_rows.
int make_map(CUtensorMap *map, const float *p, int64_t rows, int64_t k, int64_t ld, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = encoder(&enc);
    if (rc) return rc;
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * (int64_t)sizeof(float))};
    const cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           TC_BK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TRSM_SUCCESS : TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidValue;
}

int split(const float *src, int64_t ks, int64_t R, int64_t Kc, float *hi, float *lo, int64_t ldd, cudaStream_t st) {
    const dim3 grid((unsigned)((R + 31) / 32), (unsigned)((Kc + 31) / 32));
    split_tf32_kernel<<<grid, dim3(32, 8), 0, st>>>(src, ks, R, Kc, hi, lo, ldd);
    return launch_status();
}

}  // namespace

// Device address of the status word for the current device (looked up once).
int device_status_word(int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDev) return TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return cuda_status(e);
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    *out = g_status_ptr[dev];
    return TRSM_SUCCESS;
}

// Tiled tensor map of an f32 tensor (rank <= 5, dims innermost first,
// strides in bytes for dims 1..rank-1), optionally with the 128-byte
// shared-memory swizzle.  Out-of-range elements load as zero.
int encode_f32_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                   const uint32_t *box, bool swizzle128) {
    if (rank < 1 || rank > 5) return TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    const int rc = encoder(&enc);
    if (rc) return rc;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, e,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TRSM_SUCCESS : TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidValue;
}

// Workspace of the tensor-core products, 256-byte aligned regions:
//   a_hi, a_lo    the A operand (L panel, m x nb; or D_t^-1), K-major
//   x_hi, x_lo    the X operand (n x nb), K-major
//   xs_hi, xs_lo  X_t as split by the apply's epilogue for the next update
struct TcPanels {
    float *a_hi, *a_lo, *x_hi, *x_lo, *xs_hi, *xs_lo;
};

static TcPanels tc_layout(void *panels, int64_t m, int64_t n, int64_t nb) {
    TcPanels p;
    char *c = static_cast<char *>(panels);
    const size_t A = round256(m * nb * 4), X = round256(n * nb * 4);
    p.a_hi = reinterpret_cast<float *>(c);
    p.a_lo = reinterpret_cast<float *>(c + A);
    p.x_hi = reinterpret_cast<float *>(c + 2 * A);
    p.x_lo = reinterpret_cast<float *>(c + 2 * A + X);
    p.xs_hi = reinterpret_cast<float *>(c + 2 * A + 2 * X);
    p.xs_lo = reinterpret_cast<float *>(c + 2 * A + 3 * X);
    return p;
}

size_t tc_panel_bytes(int64_t m, int64_t n, int64_t nb) {
    const size_t per_block = (size_t)(2 * round256(m * nb * 4) + 4 * round256(n * nb * 4));
    const size_t fused = tc_fused_usable(m, n, nb) ? tc_fused_bytes(m, n, nb) : 0;
    return per_block > fused ? per_block : fused;
}

bool tc_update_usable(int64_t M, int64_t N, int64_t K) {
    // boxes never larger than the tensors they read
    return M >= TC_BM && N >= TC_BN && K >= TC_BK && K % TC_BK == 0;
}

bool tc_apply_usable(int64_t mb, int64_t N) {
    // enough output tiles to occupy the GPU; with fewer the FMA-pipe apply,
    // which has smaller tiles, finishes first (measured on GB300)
    const int64_t tiles = ((mb + TC_BM - 1) / TC_BM) * ((N + TC_BN - 1) / TC_BN);
    return tc_update_usable(mb, N, mb) && tiles >= 48;
}

namespace {

int split_rows(const float *src, int64_t ks, int64_t R, int64_t Kc, float *hi, float *lo, int64_t ldd,
               cudaStream_t st) {
    const bool v4 = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(hi) |
                      reinterpret_cast<uintptr_t>(lo)) & 15) == 0 && ks % 4 == 0 && Kc % 4 == 0 && ldd % 4 == 0;
    if (v4) {
        const int64_t k4 = Kc / 4;
        const dim3 grid((unsigned)((k4 + 127) / 128), (unsigned)(R < 65535 ? R : 65535));
        split_rows_tf32_v4_kernel<<<grid, 128, 0, st>>>(reinterpret_cast<const float4 *>(src), ks / 4, R, k4,
                                                        reinterpret_cast<float4 *>(hi), reinterpret_cast<float4 *>(lo),
                                                        ldd / 4);
        return launch_status();
    }
    const dim3 grid((unsigned)((Kc + 127) / 128), (unsigned)(R < 65535 ? R : 65535));
    split_rows_tf32_kernel<<<grid, 128, 0, st>>>(src, ks, R, Kc, hi, lo, ldd);
    return launch_status();
}

// The products run on CTA pairs (tc_gemm_pair_kernel): 256-row output
// tiles, each CTA loading 128 rows of A and of X.
constexpr int kTcRowsPerTile = TC2_PAIR_M;
constexpr int kTcXBox = TC_BN / 2;

int sm_count() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        sms = v > 0 ? v : 152;
    }
    return sms;
}

// Problem q of a launch: tensor maps over the K-major head/tail buffers of A
// (a_rows rows) and X (x_rows rows), row stride ld floats, K extent g.K (the
// loads zero-fill past it).  Row extents may exceed g.M / g.N (padded
// buffers): rows past them only feed outputs the epilogue discards.
int tc_problem(TcProblem &q, const float *a_hi, const float *a_lo, int64_t a_rows, const float *x_hi,
               const float *x_lo, int64_t x_rows, int64_t ld, const TcArgs &g) {
    int rc;
    if ((rc = make_map(&q.a_hi, a_hi, a_rows, g.K, ld, TC_BM))) return rc;
    if ((rc = make_map(&q.a_lo, a_lo, a_rows, g.K, ld, TC_BM))) return rc;
    if ((rc = make_map(&q.x_hi, x_hi, x_rows, g.K, ld, kTcXBox))) return rc;
    if ((rc = make_map(&q.x_lo, x_lo, x_rows, g.K, ld, kTcXBox))) return rc;
    q.g = g;
    q.tiles_m = (int)((g.M + kTcRowsPerTile - 1) / kTcRowsPerTile);
    q.tiles_n = (int)((g.N + TC_BN - 1) / TC_BN);
    q.nk = (int)((g.K + TC_BK - 1) / TC_BK);
    return TRSM_SUCCESS;
}

static_assert(sizeof(TcLaunch) <= 4096, "kernel parameters");

// One persistent launch over the tiles of P.p[0 .. np-1].
int tc_launch(TcLaunch &P, int np, cudaStream_t st) {
    int rc;
    if ((rc = device_status_word(&P.status))) return rc;
    P.np = np;
    int64_t tiles = 0;
    for (int i = 0; i < np; ++i) {
        P.p[i].tile_begin = (int)tiles;
        tiles += (int64_t)P.p[i].tiles_m * P.p[i].tiles_n;
    }
    if (tiles == 0) return TRSM_SUCCESS;
    if (tiles > INT32_MAX) return TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidValue;
    P.ntiles = (int)tiles;
    static int pairs = 0;  // CTA pairs resident at once (one CTA per SM)
    if (pairs == 0) {
        const cudaError_t e =
            cudaFuncSetAttribute(tc_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC2_SMEM);
        if (e != cudaSuccess) return cuda_status(e);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(sm_count() & ~1));
        cfg.blockDim = dim3(192);
        cfg.dynamicSmemBytes = TC2_SMEM;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = sm_count() / 2;
        }
        pairs = n;
    }
    const unsigned ctas = 2u * (unsigned)(tiles < pairs ? tiles : pairs);  // persistent
    tc_gemm_pair_kernel<<<ctas, 192, TC2_SMEM, st>>>(P);
    return launch_status();
}

int launch_tc(const float *a_hi, const float *a_lo, const float *x_hi, const float *x_lo, const TcArgs &g,
              cudaStream_t st) {
    TcLaunch P;
    const int rc = tc_problem(P.p[0], a_hi, a_lo, g.M, x_hi, x_lo, g.N, g.K, g);
    return rc ? rc : tc_launch(P, 1, st);
}

TcArgs tc_args(int64_t M, int64_t N, int64_t K, float *C, int64_t ldc) {
    TcArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.C = C;
    g.ldc = ldc;
    g.beta = 0.f;
    g.beta_im = 0.f;
    g.gamma = -1.f;
    g.gamma_im = 0.f;
    g.beta_zero = 0;
    g.a_lower = 0;
    g.a_upper = 0;
    g.cplx = 0;
    g.xmode = 0;
    g.xhi = g.xlo = nullptr;
    g.ldxs = 0;
    g.xrows = M;
    return g;
}

}  // namespace

// C (M x N, column-major ldc) = beta*C - L_panel (M x K, column-major lda) *
// X (K x N), through the TF32 head/tail panels in `panels` (tc_panel_bytes(
// Mmax, N, K) bytes, 256-byte aligned).  X is either the row-major panel X
// (ldx), split here, or -- X == nullptr -- the split copy that tc_apply_f32
// left in the panels.
int tc_update_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *X, int64_t ldx,
                  float *C, int64_t ldc, float beta, int64_t Mmax, void *panels, cudaStream_t st) {
    const TcPanels p = tc_layout(panels, Mmax, N, K);
    int rc = split(A, lda, M, K, p.a_hi, p.a_lo, K, st);  // L panel rows, K-major
    if (rc) return rc;
    const float *xh = p.xs_hi, *xl = p.xs_lo;
    if (X) {
        if ((rc = split(X, ldx, N, K, p.x_hi, p.x_lo, K, st))) return rc;  // X_t columns, K-major
        xh = p.x_hi;
        xl = p.x_lo;
    }
    TcArgs g = tc_args(M, N, K, C, ldc);
    g.beta = beta;
    return launch_tc(p.a_hi, p.a_lo, xh, xl, g, st);
}

// c64 panels: A' (Mmax x 2nb), X' (2N x 2nb), and the split X_t' the complex
// apply leaves for the update, head and tail each.
struct TcPanelsC64 {
    float *a_hi, *a_lo, *x_hi, *x_lo, *xs_hi, *xs_lo;
};

static TcPanelsC64 tc_layout_c64(void *panels, int64_t m, int64_t n, int64_t nb) {
    TcPanelsC64 p;
    char *c = static_cast<char *>(panels);
    const size_t A = round256(m * 2 * nb * 4), X = round256(2 * n * 2 * nb * 4);
    p.a_hi = reinterpret_cast<float *>(c);
    p.a_lo = reinterpret_cast<float *>(c + A);
    p.x_hi = reinterpret_cast<float *>(c + 2 * A);
    p.x_lo = reinterpret_cast<float *>(c + 2 * A + X);
    p.xs_hi = reinterpret_cast<float *>(c + 2 * A + 2 * X);
    p.xs_lo = reinterpret_cast<float *>(c + 2 * A + 3 * X);
    return p;
}

size_t tc_panel_bytes_c64(int64_t m, int64_t n, int64_t nb) {
    const size_t per_block = (size_t)(2 * round256(m * 2 * nb * 4) + 4 * round256(2 * n * 2 * nb * 4));
    const size_t fused = tc_fused_usable_c64(m, n, nb) ? tc_fused_bytes_c64(m, n, nb) : 0;
    return per_block > fused ? per_block : fused;
}

// c64 trailing update C = beta*C - A X (A column-major lda, all complex) as
// one real product of M x 2N x 2K on the tensor cores (see split_c64_*).
// X is the row-major panel (ldx), split here, or -- X == nullptr -- the split
// copy tc_apply_c64 left in the panels (tc_panel_bytes_c64(Mmax, N, K)).
int tc_update_c64(int64_t M, int64_t N, int64_t K, const float2 *A, int64_t lda, const float2 *X, int64_t ldx,
                  float2 *C, int64_t ldc, float2 beta, int64_t Mmax, void *panels, cudaStream_t st) {
    const TcPanelsC64 p = tc_layout_c64(panels, Mmax, N, K);
    split_c64_a_kernel<<<dim3((unsigned)((M + 31) / 32), (unsigned)((K + 31) / 32)), dim3(32, 8), 0, st>>>(
        A, lda, M, K, p.a_hi, p.a_lo);
    int rc = launch_status();
    if (rc) return rc;
    const float *xh = p.xs_hi, *xl = p.xs_lo;
    if (X) {
        split_c64_x_kernel<<<dim3((unsigned)((N + 31) / 32), (unsigned)((K + 31) / 32)), dim3(32, 8), 0, st>>>(
            X, ldx, K, N, p.x_hi, p.x_lo);
        if ((rc = launch_status())) return rc;
        xh = p.x_hi;
        xl = p.x_lo;
    }
    TcArgs g = tc_args(M, 2 * N, 2 * K, reinterpret_cast<float *>(C), 2 * ldc);
    g.beta = beta.x;
    g.beta_im = beta.y;
    g.cplx = 1;
    return launch_tc(p.a_hi, p.a_lo, xh, xl, g, st);
}

bool tc_apply_usable_c64(int64_t mb, int64_t N) {
    const int64_t tiles = ((mb + TC_BM - 1) / TC_BM) * ((2 * N + TC_BN - 1) / TC_BN);
    return tc_update_usable(mb, 2 * N, 2 * mb) && tiles >= 48;
}

// Complex block apply on the tensor cores: X_t = gamma * D_t^-1 R_t over R_t
// (block row of B, column-major ldb), D_t^-1 the column-major lower-
// triangular block Wt (ld nb); real form with interleaved K' so the
// triangular K range stays a prefix.  With emit_split the epilogue leaves
// X_t' split for tc_update_c64 (X == nullptr).
int tc_apply_c64(int64_t mb, int64_t N, const float2 *Wt, int64_t nb, float2 *Bt, int64_t ldb, float2 gamma,
                 int64_t Mmax, void *panels, bool emit_split, cudaStream_t st) {
    const TcPanelsC64 p = tc_layout_c64(panels, Mmax, N, nb);
    split_c64_ai_kernel<<<dim3((unsigned)((mb + 31) / 32), (unsigned)((mb + 31) / 32)), dim3(32, 8), 0, st>>>(
        Wt, nb, mb, mb, p.a_hi, p.a_lo, 2 * mb);
    int rc = launch_status();
    if (rc) return rc;
    split_c64_xi_kernel<<<dim3((unsigned)((mb + 127) / 128), (unsigned)(N < 65535 ? N : 65535)), 128, 0, st>>>(
        Bt, ldb, mb, N, p.x_hi, p.x_lo, 2 * mb);
    if ((rc = launch_status())) return rc;
    TcArgs g = tc_args(mb, 2 * N, 2 * mb, reinterpret_cast<float *>(Bt), 2 * ldb);
    g.beta_zero = 1;
    g.gamma = gamma.x;
    g.gamma_im = gamma.y;
    g.a_lower = 2;
    g.cplx = 1;
    if (emit_split) {
        g.xhi = p.xs_hi;
        g.xlo = p.xs_lo;
        g.ldxs = 2 * nb;
    }
    return launch_tc(p.a_hi, p.a_lo, p.x_hi, p.x_lo, g, st);
}

// Block apply on the tensor cores: X_t = gamma * D_t^-1 R_t, written over
// R_t (its block row of B: mb x N, column-major ldb); D_t^-1 is the
// column-major lower-triangular block Wt (ld nb).  With emit_split the
// epilogue also leaves X_t split, K-major, for tc_update_f32 (X == nullptr).
int tc_apply_f32(int64_t mb, int64_t N, const float *Wt, int64_t nb, float *Bt, int64_t ldb, float gamma,
                 int64_t Mmax, void *panels, bool emit_split, cudaStream_t st) {
    const TcPanels p = tc_layout(panels, Mmax, N, nb);
    int rc = split(Wt, nb, mb, mb, p.a_hi, p.a_lo, mb, st);  // rows of D_t^-1, K-major
    if (!rc) rc = split_rows(Bt, ldb, N, mb, p.x_hi, p.x_lo, mb, st);  // columns of R_t
    if (rc) return rc;
    TcArgs g = tc_args(mb, N, mb, Bt, ldb);
    g.beta_zero = 1;
    g.gamma = gamma;
    g.a_lower = 1;
    if (emit_split) {
        g.xhi = p.xs_hi;
        g.xlo = p.xs_lo;
        g.ldxs = nb;
    }
    return launch_tc(p.a_hi, p.a_lo, p.x_hi, p.x_lo, g, st);
}

// ---------------------------------------------------------------------------
// Look-ahead form of the f32 blocked solve.  With W_t = L_panel_t D_t^-1
// (L_panel_t: the rows of L below block t, in its columns) the update of
// block t reads the block row R_t itself,
//     B_below -= W_t R_t,
// so X_t = D_t^-1 R_t is off the path from one block to the next.  Launch t
// computes, as one tile list:
//   the update of block t      (m - r0 - nb) x n x nb, its first nb rows
//                              (R_{t+1}, final now) also stored split: the
//                              X operand of the next update and apply,
//   W_{t+1} for the next step  (W_{t+1}^T = D_{t+1}^-T L_panel_{t+1}^T,
//                              nb x (m - r1 - nb) x nb, upper-triangular A,
//                              stored split: the A operand of update t+1),
//   the apply of block t-1     nb x n x nb, lower-triangular A, over R_{t-1},
// and the last launch both remaining applies.  The apply thus fills the
// rounds of the update instead of running in under two rounds of its own,
// no split copy of X_t is written, and no pass splits the block rows.  W_0
// and the split of R_0 are made before the first step.  Extra work: the W_t products, nb/n of the updates' flops (half of it
// with the triangular K range).
//
// Workspace (256-byte aligned regions, rows padded for the TMA boxes):
//   wp[2]   W_t head/tail, RA x nb (A operand of the update; double buffer)
//   lp[2]   L_panel_b head/tail, RA x nb (X operand of W_b^T; double buffer:
//           block b's copy is made on a side stream while launch b-2 runs)
//   xs[3]   R_t head/tail, RX x nb (X operand of update t and apply t; launch
//           t reads R_t and R_{t-1} and writes R_{t+1}: three buffers)
//   d0      D^-1 rows (apply), head/tail, nb x nb
//   d1[2]   D_b^-T rows (W product; made with lp[b & 1]), head/tail, nb x nb
// with RA = m and RX = n rounded up to 256 rows.
// ---------------------------------------------------------------------------
namespace {

// Below this many right-hand sides the W_t products (nb/n of the update
// flops) and the narrow tiles make the per-block flow the faster one.
constexpr int64_t kTcFusedMinN = 256;

struct TcFused {
    float *wp_hi[2], *wp_lo[2], *lp_hi[2], *lp_lo[2], *xs_hi[3], *xs_lo[3], *d0_hi, *d0_lo, *d1_hi[2], *d1_lo[2];
    int64_t ra, rx;
};

int64_t round_rows(int64_t r) { return (r + 255) / 256 * 256; }

// Columns a product must cover: all n, or with a lower-triangular identity
// right-hand side (tri) only the first `upto` of them.
int64_t tri_cols(bool tri, int64_t n, int64_t upto) { return (tri && upto < n) ? upto : n; }

TcFused tc_fused_layout(void *panels, int64_t m, int64_t n, int64_t nb) {
    TcFused f;
    f.ra = round_rows(m);
    f.rx = round_rows(n);
    const size_t A = round256(f.ra * nb * 4), X = round256(f.rx * nb * 4), D = round256(nb * nb * 4);
    char *c = static_cast<char *>(panels);
    auto take = [&](size_t bytes) {
        float *p = reinterpret_cast<float *>(c);
        c += bytes;
        return p;
    };
    for (int i = 0; i < 2; ++i) {
        f.wp_hi[i] = take(A);
        f.wp_lo[i] = take(A);
    }
    for (int i = 0; i < 2; ++i) {
        f.lp_hi[i] = take(A);
        f.lp_lo[i] = take(A);
    }
    for (int i = 0; i < 3; ++i) {
        f.xs_hi[i] = take(X);
        f.xs_lo[i] = take(X);
    }
    f.d0_hi = take(D);
    f.d0_lo = take(D);
    for (int i = 0; i < 2; ++i) {
        f.d1_hi[i] = take(D);
        f.d1_lo[i] = take(D);
    }
    return f;
}

// The operands of block b's W product, which depend on L and D_b^-1 only:
// its L panel and D_b^-T split into lp[b & 1], d1[b & 1].
int tc_w_splits(const TcFused &f, int64_t b, int64_t m, int64_t nb, const float *L, int64_t lda, const float *W,
                cudaStream_t st) {
    const int64_t r1 = b * nb, rows = m - r1 - nb;
    const int rc = split(L + r1 * lda + r1 + nb, lda, rows, nb, f.lp_hi[b & 1], f.lp_lo[b & 1], nb, st);
    return rc ? rc : split_rows(W + b * nb * nb, nb, nb, nb, f.d1_hi[b & 1], f.d1_lo[b & 1], nb, st);
}

// The W_{t+1}^T product of launch t (and of the preparation, t = -1): block
// b = t + 1, from its split operands, emitting W_b.
int tc_w_problem(TcProblem &q, const TcFused &f, int64_t b, int64_t m, int64_t nb) {
    const int64_t r1 = b * nb, rows = m - r1 - nb;
    TcArgs g = tc_args(nb, rows, nb, nullptr, 0);
    g.beta_zero = 1;
    g.gamma = 1.f;
    g.a_upper = 1;
    g.xhi = f.wp_hi[b & 1];
    g.xlo = f.wp_lo[b & 1];
    g.ldxs = nb;
    return tc_problem(q, f.d1_hi[b & 1], f.d1_lo[b & 1], nb, f.lp_hi[b & 1], f.lp_lo[b & 1], f.ra, nb, g);
}

// The apply of block b over its block row (R_b split in xs[b % 3]); the D_b^-1
// rows go to (dh, dl).
int tc_x_problem(TcProblem &q, const TcFused &f, int64_t b, int64_t m, int64_t n, int64_t nb, const float *W,
                 float *B, int64_t ldb, float gamma, float *dh, float *dl, cudaStream_t st) {
    const int64_t r0 = b * nb, mb = (m - r0 < nb) ? m - r0 : nb;
    const int rc = split(W + b * nb * nb, nb, mb, mb, dh, dl, nb, st);  // rows of D_b^-1, K-major
    if (rc) return rc;
    TcArgs g = tc_args(mb, n, mb, B + r0, ldb);
    g.beta_zero = 1;
    g.gamma = gamma;
    g.a_lower = 1;
    return tc_problem(q, dh, dl, nb, f.xs_hi[b % 3], f.xs_lo[b % 3], f.rx, nb, g);
}

}  // namespace

bool tc_fused_usable(int64_t m, int64_t n, int64_t nb) {
    if (nb != 128 && nb != 256 && nb != 512) return false;
    const int64_t tb = (m + nb - 1) / nb, mb_last = m - (tb - 1) * nb;
    const int64_t tiles = ((m + TC_BM - 1) / TC_BM) * ((n + TC_BN - 1) / TC_BN);
    return tb >= 2 && mb_last >= TC_BK && n >= kTcFusedMinN && tiles < INT32_MAX;
}

size_t tc_fused_bytes(int64_t m, int64_t n, int64_t nb) {
    const int64_t ra = round_rows(m), rx = round_rows(n);
    return (size_t)(8 * round256(ra * nb * 4) + 6 * round256(rx * nb * 4) + 6 * round256(nb * nb * 4));
}

// The side stream of the L-panel splits: the persistent tensor-core launch
// leaves room on every SM for a split CTA, and the splits (HBM-bound, on L
// and the inverted blocks only) run beside the launch before the one that
// needs them.  launched[t & 1] marks launch t done, split[b & 1] block b's
// operands ready; the side stream starts after everything already on st.
namespace {

// One side stream and its events per (device, caller stream), created on
// first use and kept for the life of the process; a solve holds its slot
// (the lock) from acquire to release, so the event records of two solves
// never interleave.  Reuse across solves is safe: every wait of a solve
// refers to an event recorded earlier in the same solve.
struct SideSlot : TcSide {
    std::mutex mu;
};
std::mutex g_side_map_mu;
std::map<std::pair<int, cudaStream_t>, SideSlot *> g_side_slots;

void side_destroy(TcSide &side) {
    for (int i = 0; i < 2; ++i) {
        if (side.launched[i]) cudaEventDestroy(side.launched[i]);
        if (side.split[i]) cudaEventDestroy(side.split[i]);
    }
    if (side.start) cudaEventDestroy(side.start);
    if (side.s) cudaStreamDestroy(side.s);
    side.s = nullptr;
    side.launched[0] = side.launched[1] = side.split[0] = side.split[1] = side.start = nullptr;
}

}  // namespace

int tc_side_acquire(cudaStream_t st, TcSide **out) {
    *out = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    SideSlot *slot = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_side_map_mu);
        SideSlot *&p = g_side_slots[{dev, st}];
        if (!p) p = new SideSlot;
        slot = p;
    }
    slot->mu.lock();
    TcSide &side = *slot;
    if (!side.s) {
        e = cudaStreamCreateWithFlags(&side.s, cudaStreamNonBlocking);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&side.launched[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&side.split[i], cudaEventDisableTiming);
        }
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&side.start, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            side_destroy(side);
            slot->mu.unlock();
            return cuda_status(e);
        }
    }
    // the side stream starts after everything already queued on st
    e = cudaEventRecord(side.start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side.s, side.start, 0);
    if (e != cudaSuccess) {
        slot->mu.unlock();
        return cuda_status(e);
    }
    *out = &side;
    return TRSM_SUCCESS;
}

void tc_side_release(TcSide *side) {
    if (side) static_cast<SideSlot *>(side)->mu.unlock();
}

// W_0 = L_panel_0 D_0^-1 and the split of R_0, before step 0; block 1's W
// operands too (launch 0 needs them before the side stream could make them).
// This launch counts as launch -1 for the side stream (it reads block 0's
// operand buffers, which block 2's overwrite).
int tc_fused_prepare_side(int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W,
                          const float *B, int64_t ldb, void *panels, cudaStream_t st, TcSide *side, bool tri) {
    const TcFused f = tc_fused_layout(panels, m, n, nb);
    // columns of R_0 (tri: the first two blocks, all update 0 reads)
    int rc = split_rows(B, ldb, tri_cols(tri, n, 2 * nb), nb, f.xs_hi[0], f.xs_lo[0], nb, st);
    if (!rc) rc = tc_w_splits(f, 0, m, nb, L, lda, W, st);
    if (!rc && 2 * nb < m) rc = tc_w_splits(f, 1, m, nb, L, lda, W, st);
    if (rc) return rc;
    TcLaunch P;
    rc = tc_w_problem(P.p[0], f, 0, m, nb);
    if (!rc) rc = tc_launch(P, 1, st);
    if (!rc && side) rc = cuda_status(cudaEventRecord(side->launched[1], st));
    return rc;
}

// Step t: one launch of update t (leaving R_{t+1} split), W_{t+1} and apply
// t-1; the last step: apply t and apply t-1.  alpha enters through block 0.
// With `side`, block t+2's W operands are made on the side stream once
// launch t-1 is done (their buffers were last read by it), and launch t
// waits for block t+1's.
int tc_fused_step_side(int64_t t, int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W,
                       float *B, int64_t ldb, float alpha, void *panels, cudaStream_t st, TcSide *side, bool tri) {
    const TcFused f = tc_fused_layout(panels, m, n, nb);
    const int64_t tb = (m + nb - 1) / nb, r0 = t * nb;
    int rc;
    cudaError_t e = cudaSuccess;
    if (side && r0 + 3 * nb < m) {  // block t+2 has rows below it
        // launch t-1 (t = 0: the preparation's) last read these buffers
        if ((e = cudaStreamWaitEvent(side->s, side->launched[(t + 1) & 1], 0)) != cudaSuccess) return cuda_status(e);
        if ((rc = tc_w_splits(f, t + 2, m, nb, L, lda, W, side->s))) return rc;
        if ((e = cudaEventRecord(side->split[(t + 2) & 1], side->s)) != cudaSuccess) return cuda_status(e);
    }
    TcLaunch P;
    int np = 0;
    if (t + 1 < tb) {
        TcArgs g = tc_args(m - r0 - nb, tri_cols(tri, n, (t + 2) * nb), nb, B + r0 + nb, ldb);
        g.beta = t == 0 ? alpha : 1.f;
        g.gamma = t == 0 ? -alpha : -1.f;
        g.xhi = f.xs_hi[(t + 1) % 3];
        g.xlo = f.xs_lo[(t + 1) % 3];
        g.ldxs = nb;
        g.xrows = nb;
        if ((rc = tc_problem(P.p[np++], f.wp_hi[t & 1], f.wp_lo[t & 1], f.ra, f.xs_hi[t % 3], f.xs_lo[t % 3], f.rx,
                             nb, g)))
            return rc;
        if (r0 + 2 * nb < m) {  // block t+1 has rows below it: its W product
            if (!side && (rc = tc_w_splits(f, t + 1, m, nb, L, lda, W, st))) return rc;
            if (side && t + 1 >= 2 && (e = cudaStreamWaitEvent(st, side->split[(t + 1) & 1], 0)) != cudaSuccess)
                return cuda_status(e);
            if ((rc = tc_w_problem(P.p[np++], f, t + 1, m, nb))) return rc;
        }
    } else if ((rc = tc_x_problem(P.p[np++], f, t, m, tri_cols(tri, n, (t + 1) * nb), nb, W, B, ldb,
                                  t == 0 ? alpha : 1.f, f.d1_hi[0], f.d1_lo[0], st))) {
        return rc;
    }
    if (t >= 1 && (rc = tc_x_problem(P.p[np++], f, t - 1, m, tri_cols(tri, n, t * nb), nb, W, B, ldb,
                                     t == 1 ? alpha : 1.f, f.d0_hi, f.d0_lo, st)))
        return rc;
    if ((rc = tc_launch(P, np, st))) return rc;
    if (side && (e = cudaEventRecord(side->launched[t & 1], st)) != cudaSuccess) return cuda_status(e);
    if (tri && (t + 2) * nb < n) {
        // update t+1 reads R_{t+1} over its first (t+3) nb columns; the
        // epilogue above split the first (t+2) nb, the next block of them is
        // zero (those columns of the identity start below block t+1)
        const int64_t j0 = (t + 2) * nb, rows = (n - j0 < nb) ? n - j0 : nb;
        const size_t off = (size_t)(j0 * nb), bytes = (size_t)(rows * nb) * sizeof(float);
        if ((e = cudaMemsetAsync(f.xs_hi[(t + 1) % 3] + off, 0, bytes, st)) != cudaSuccess) return cuda_status(e);
        if ((e = cudaMemsetAsync(f.xs_lo[(t + 1) % 3] + off, 0, bytes, st)) != cudaSuccess) return cuda_status(e);
    }
    return TRSM_SUCCESS;
}

int tc_fused_prepare(int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W, const float *B,
                     int64_t ldb, void *panels, cudaStream_t st, bool tri) {
    return tc_fused_prepare_side(m, n, nb, L, lda, W, B, ldb, panels, st, nullptr, tri);
}

int tc_fused_step(int64_t t, int64_t m, int64_t n, int64_t nb, const float *L, int64_t lda, const float *W,
                  float *B, int64_t ldb, float alpha, void *panels, cudaStream_t st, bool tri) {
    return tc_fused_step_side(t, m, n, nb, L, lda, W, B, ldb, alpha, panels, st, nullptr, tri);
}

// ---------------------------------------------------------------------------
// The look-ahead form for c64, in real form with interleaved K throughout
// (k' = 2k real part, 2k + 1 imaginary part), so that the update and the
// apply read the same split block row:
//   A' of W_t      row i = [Re W(i,0), Im W(i,0), Re W(i,1), ...]   (ra x 2nb)
//   X' of R_t      rows 2j, 2j+1 of column j, interleaved (xmode 1)  (2rx x 2nb)
//   X' of L_panel^T rows 2i, 2i+1 of panel row i, interleaved        (2ra x 2nb)
//   A' of D^-1 / D^-T rows, interleaved                              (nb x 2nb)
// The W_{t+1}^T product leaves W_{t+1} transposed in A' layout (xmode 2);
// update t leaves R_{t+1} in X' layout (xmode 1).
// ---------------------------------------------------------------------------
namespace {

struct TcFusedC64 {
    float *wp_hi[2], *wp_lo[2], *lp_hi, *lp_lo, *xs_hi[3], *xs_lo[3], *d0_hi, *d0_lo, *d1_hi, *d1_lo;
    int64_t ra, rx;
};

TcFusedC64 tc_fused_layout_c64(void *panels, int64_t m, int64_t n, int64_t nb) {
    TcFusedC64 f;
    f.ra = round_rows(m);
    f.rx = round_rows(n);
    const size_t A = round256(f.ra * 2 * nb * 4), L = round256(2 * f.ra * 2 * nb * 4),
                 X = round256(2 * f.rx * 2 * nb * 4), D = round256(nb * 2 * nb * 4);
    char *c = static_cast<char *>(panels);
    auto take = [&](size_t bytes) {
        float *p = reinterpret_cast<float *>(c);
        c += bytes;
        return p;
    };
    for (int i = 0; i < 2; ++i) {
        f.wp_hi[i] = take(A);
        f.wp_lo[i] = take(A);
    }
    f.lp_hi = take(L);
    f.lp_lo = take(L);
    for (int i = 0; i < 3; ++i) {
        f.xs_hi[i] = take(X);
        f.xs_lo[i] = take(X);
    }
    f.d0_hi = take(D);
    f.d0_lo = take(D);
    f.d1_hi = take(D);
    f.d1_lo = take(D);
    return f;
}

int tc_w_problem_c64(TcProblem &q, const TcFusedC64 &f, int64_t b, int64_t m, int64_t nb, const float2 *L,
                     int64_t lda, const float2 *W, cudaStream_t st) {
    const int64_t r1 = b * nb, rows = m - r1 - nb;
    split_c64_xt_kernel<<<dim3((unsigned)((rows + 31) / 32), (unsigned)((nb + 31) / 32)), dim3(32, 8), 0, st>>>(
        L + r1 * lda + r1 + nb, lda, rows, nb, f.lp_hi, f.lp_lo, 2 * nb);
    int rc = launch_status();
    // rows of D_b^-T, interleaved: column r of the column-major D_b^-1 as float pairs
    if (!rc) rc = split_rows(reinterpret_cast<const float *>(W + b * nb * nb), 2 * nb, nb, 2 * nb, f.d1_hi, f.d1_lo,
                             2 * nb, st);
    if (rc) return rc;
    TcArgs g = tc_args(nb, 2 * rows, 2 * nb, nullptr, 0);
    g.beta_zero = 1;
    g.gamma = 1.f;
    g.a_upper = 2;
    g.cplx = 1;
    g.xhi = f.wp_hi[b & 1];
    g.xlo = f.wp_lo[b & 1];
    g.ldxs = 2 * nb;
    g.xmode = 2;
    return tc_problem(q, f.d1_hi, f.d1_lo, nb, f.lp_hi, f.lp_lo, 2 * f.ra, 2 * nb, g);
}

int tc_x_problem_c64(TcProblem &q, const TcFusedC64 &f, int64_t b, int64_t m, int64_t n, int64_t nb,
                     const float2 *W, float2 *B, int64_t ldb, float2 gamma, float *dh, float *dl, cudaStream_t st) {
    const int64_t r0 = b * nb, mb = (m - r0 < nb) ? m - r0 : nb;
    split_c64_ai_kernel<<<dim3((unsigned)((mb + 31) / 32), (unsigned)((mb + 31) / 32)), dim3(32, 8), 0, st>>>(
        W + b * nb * nb, nb, mb, mb, dh, dl, 2 * nb);
    const int rc = launch_status();
    if (rc) return rc;
    TcArgs g = tc_args(mb, 2 * n, 2 * mb, reinterpret_cast<float *>(B + r0), 2 * ldb);
    g.beta_zero = 1;
    g.gamma = gamma.x;
    g.gamma_im = gamma.y;
    g.a_lower = 2;
    g.cplx = 1;
    return tc_problem(q, dh, dl, nb, f.xs_hi[b % 3], f.xs_lo[b % 3], 2 * f.rx, 2 * nb, g);
}

}  // namespace

bool tc_fused_usable_c64(int64_t m, int64_t n, int64_t nb) {
    // The same shapes as f32, up to n = 8192.  Measured on GB300 (same box,
    // NB 512): m = n = 8192 9.09 ms against 9.66 per block, m = n = 16384
    // 65.1 against 63.9 -- once the split block row (2n x 2NB floats, head
    // and tail: 268 MB at n = 16384) is twice the L2, the launch's extra
    // panels of that size (R_{t+1} written, the L panel's X' read) cost what
    // the folded apply saves.
    return n <= 8192 && tc_fused_usable(m, n, nb);
}

size_t tc_fused_bytes_c64(int64_t m, int64_t n, int64_t nb) {
    const int64_t ra = round_rows(m), rx = round_rows(n);
    return (size_t)(4 * round256(ra * 2 * nb * 4) + 2 * round256(2 * ra * 2 * nb * 4) +
                    6 * round256(2 * rx * 2 * nb * 4) + 4 * round256(nb * 2 * nb * 4));
}

int tc_fused_prepare_c64(int64_t m, int64_t n, int64_t nb, const float2 *L, int64_t lda, const float2 *W,
                         const float2 *B, int64_t ldb, void *panels, cudaStream_t st, bool tri) {
    const TcFusedC64 f = tc_fused_layout_c64(panels, m, n, nb);
    const int64_t n0 = tri_cols(tri, n, 2 * nb);  // tri: the columns update 0 reads
    split_c64_xi_kernel<<<dim3((unsigned)((nb + 127) / 128), (unsigned)(n0 < 65535 ? n0 : 65535)), 128, 0, st>>>(
        B, ldb, nb, n0, f.xs_hi[0], f.xs_lo[0], 2 * nb);  // R_0, interleaved X'
    int rc = launch_status();
    if (rc) return rc;
    TcLaunch P;
    rc = tc_w_problem_c64(P.p[0], f, 0, m, nb, L, lda, W, st);
    return rc ? rc : tc_launch(P, 1, st);
}

int tc_fused_step_c64(int64_t t, int64_t m, int64_t n, int64_t nb, const float2 *L, int64_t lda, const float2 *W,
                      float2 *B, int64_t ldb, float2 alpha, void *panels, cudaStream_t st, bool tri) {
    const TcFusedC64 f = tc_fused_layout_c64(panels, m, n, nb);
    const int64_t tb = (m + nb - 1) / nb, r0 = t * nb;
    const float2 one = make_float2(1.f, 0.f);
    int rc;
    TcLaunch P;
    int np = 0;
    if (t + 1 < tb) {
        TcArgs g = tc_args(m - r0 - nb, 2 * tri_cols(tri, n, (t + 2) * nb), 2 * nb,
                           reinterpret_cast<float *>(B + r0 + nb), 2 * ldb);
        const float2 beta = t == 0 ? alpha : one;
        g.beta = beta.x;
        g.beta_im = beta.y;
        g.gamma = -beta.x;
        g.gamma_im = -beta.y;
        g.cplx = 1;
        g.xhi = f.xs_hi[(t + 1) % 3];
        g.xlo = f.xs_lo[(t + 1) % 3];
        g.ldxs = 2 * nb;
        g.xrows = nb;
        g.xmode = 1;
        if ((rc = tc_problem(P.p[np++], f.wp_hi[t & 1], f.wp_lo[t & 1], f.ra, f.xs_hi[t % 3], f.xs_lo[t % 3],
                             2 * f.rx, 2 * nb, g)))
            return rc;
        if (r0 + 2 * nb < m && (rc = tc_w_problem_c64(P.p[np++], f, t + 1, m, nb, L, lda, W, st))) return rc;
    } else if ((rc = tc_x_problem_c64(P.p[np++], f, t, m, tri_cols(tri, n, (t + 1) * nb), nb, W, B, ldb,
                                      t == 0 ? alpha : one, f.d1_hi, f.d1_lo, st))) {
        return rc;
    }
    if (t >= 1 && (rc = tc_x_problem_c64(P.p[np++], f, t - 1, m, tri_cols(tri, n, t * nb), nb, W, B, ldb,
                                         t == 1 ? alpha : one, f.d0_hi, f.d0_lo, st)))
        return rc;
    if ((rc = tc_launch(P, np, st))) return rc;
    if (tri && (t + 2) * nb < n) {
        // as for f32: the next block of R_{t+1}'s columns is zero (rows 2j,
        // 2j+1 of the interleaved panel for column j)
        const int64_t j0 = (t + 2) * nb, rows = (n - j0 < nb) ? n - j0 : nb;
        const size_t off = (size_t)(2 * j0 * 2 * nb), bytes = (size_t)(2 * rows * 2 * nb) * sizeof(float);
        cudaError_t e;
        if ((e = cudaMemsetAsync(f.xs_hi[(t + 1) % 3] + off, 0, bytes, st)) != cudaSuccess) return cuda_status(e);
        if ((e = cudaMemsetAsync(f.xs_lo[(t + 1) % 3] + off, 0, bytes, st)) != cudaSuccess) return cuda_status(e);
    }
    return TRSM_SUCCESS;
}

namespace {
std::atomic<uint32_t> g_first_wait_limit{kWaitLimit};
}  // namespace

uint32_t first_wait_limit() { return g_first_wait_limit.load(std::memory_order_relaxed); }

int set_first_wait_limit(int64_t polls) {
    g_first_wait_limit.store(polls < 0 || polls > (int64_t)kWaitLimit ? kWaitLimit : (uint32_t)polls,
                             std::memory_order_relaxed);
    return TRSM_SUCCESS;
}

int device_status(int clear) {
    int *p = nullptr;
    int rc = device_status_word(&p);
    if (rc) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_status(e);
    int v = 0;
    e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    if (clear && v) {
        const int z = 0;
        e = cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return v;
}

}  // namespace trsm
