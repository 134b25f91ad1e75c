// Host side of the tensor-core f32 trailing update: TF32 head/tail split of
// the two panels, tensor maps for the TMA loads, launch, and the device
// status word that the kernels' bounded waits report to.
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_gemm.cuh"

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
    return (size_t)(2 * round256(m * nb * 4) + 4 * round256(n * nb * 4));
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

int launch_tc(const float *a_hi, const float *a_lo, const float *x_hi, const float *x_lo, TcArgs g, cudaStream_t st) {
    CUtensorMap ma_hi, ma_lo, mx_hi, mx_lo;
    int rc;
    if ((rc = make_map(&ma_hi, a_hi, g.M, g.K, g.K, TC_BM))) return rc;
    if ((rc = make_map(&ma_lo, a_lo, g.M, g.K, g.K, TC_BM))) return rc;
    if ((rc = make_map(&mx_hi, x_hi, g.N, g.K, g.K, TC_BN))) return rc;
    if ((rc = make_map(&mx_lo, x_lo, g.N, g.K, g.K, TC_BN))) return rc;
    if ((rc = device_status_word(&g.status))) return rc;
    const cudaError_t e =
        cudaFuncSetAttribute(tc_update_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    if (e != cudaSuccess) return cuda_status(e);
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
    }
    const int64_t tiles = ((g.M + TC_BM - 1) / TC_BM) * ((g.N + TC_BN - 1) / TC_BN);
    const unsigned ctas = (unsigned)(tiles < sms ? tiles : sms);  // persistent: one CTA per SM
    tc_update_f32_kernel<<<ctas, 192, TC_SMEM, st>>>(ma_hi, ma_lo, mx_hi, mx_lo, g);
    return launch_status();
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
    g.cplx = 0;
    g.xhi = g.xlo = nullptr;
    g.ldxs = 0;
    g.status = nullptr;
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
    return (size_t)(2 * round256(m * 2 * nb * 4) + 4 * round256(2 * n * 2 * nb * 4));
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
        Wt, nb, mb, mb, p.a_hi, p.a_lo);
    int rc = launch_status();
    if (rc) return rc;
    split_c64_xi_kernel<<<dim3((unsigned)((mb + 127) / 128), (unsigned)(N < 65535 ? N : 65535)), 128, 0, st>>>(
        Bt, ldb, mb, N, p.x_hi, p.x_lo);
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
