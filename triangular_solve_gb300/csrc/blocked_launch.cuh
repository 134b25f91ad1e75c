// Host driver of the blocked path for one element type.
#pragma once

#include <algorithm>
#include <type_traits>

#include "blocked_kernels.cuh"
#include "few_rhs.cuh"
#include "gemm_sp.cuh"
#include "internal.h"
#include "tc_side.h"

namespace trsm {

// Generic GEMM: the regular tiles when they fill two waves of SMs, else
// the small tiles.
template <typename T>
static int gemm_launch(const GemmArgs<T> &g, cudaStream_t st, int nz = 1) {
    using C = GemmCfg<T, false>;
    using S = GemmCfg<T, true>;
    if (g.M <= 0 || g.N <= 0 || nz <= 0) return TRSM_SUCCESS;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
    }
    const int64_t ctas = ((g.M + C::BM - 1) / C::BM) * ((g.N + C::BN - 1) / C::BN) * nz;
    if (ctas >= 2 * sms) {
        const dim3 grid((unsigned)((g.M + C::BM - 1) / C::BM), (unsigned)((g.N + C::BN - 1) / C::BN), (unsigned)nz);
        gemm_kernel<T, false><<<grid, 256, 0, st>>>(g);
    } else {
        const dim3 grid((unsigned)((g.M + S::BM - 1) / S::BM), (unsigned)((g.N + S::BN - 1) / S::BN), (unsigned)nz);
        gemm_kernel<T, true><<<grid, 256, 0, st>>>(g);
    }
    return launch_status();
}

// Launch the single-precision GEMM with large tiles when they fill at least
// two waves of the GPU's SMs, else with the small tiles.
template <typename T>
static int sp_launch(const SpArgs &g, cudaStream_t st, int nz = 1) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 152;
    }
    using Big = SpTile<T, false>;
    const int64_t big_ctas = ((g.M + Big::BM - 1) / Big::BM) * ((g.N + Big::BN - 1) / Big::BN) * nz;
    auto go = [&](auto tile_tag, auto kern) -> int {
        using Tl = decltype(tile_tag);
        if (Tl::SMEM > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Tl::SMEM);
            if (e != cudaSuccess) return cuda_status(e);
        }
        const dim3 grid((unsigned)((g.M + Tl::BM - 1) / Tl::BM), (unsigned)((g.N + Tl::BN - 1) / Tl::BN),
                        (unsigned)nz);
        kern<<<grid, 256, Tl::SMEM, st>>>(g);
        return launch_status();
    };
    if (big_ctas >= 2 * sms) return go(SpTile<T, false>{}, sp_update_kernel<T, false>);
    return go(SpTile<T, true>{}, sp_update_kernel<T, true>);
}

// Trailing update C = beta*C - A X (A column-major, X row-major panel).
template <typename T>
static int update_launch(int64_t M, int64_t N, int64_t K, const T *A, int64_t lda, const T *X, int64_t ldx,
                         T *C, int64_t ldc, T beta, T minus_one, cudaStream_t st, int64_t Mmax = 0,
                         void *tc_panels = nullptr) {
    if (M <= 0 || N <= 0) return TRSM_SUCCESS;
    if constexpr (std::is_same<T, float>::value) {
        if (tc_panels && tc_update_usable(M, N, K))
            return tc_update_f32(M, N, K, A, lda, X, ldx, C, ldc, beta, Mmax, tc_panels, st);
    }
    if constexpr (std::is_same<T, float2>::value) {
        if (tc_panels && tc_update_usable(M, 2 * N, 2 * K))
            return tc_update_c64(M, N, K, A, lda, X, ldx, C, ldc, beta, Mmax, tc_panels, st);
    }
    if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value) {
        const bool aligned = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) &&
                             ((lda * (int64_t)sizeof(T)) % 16 == 0);
        if (aligned) {
            SpArgs g;
            g.M = M; g.N = N; g.K = K;
            g.A = A; g.lda = lda;
            g.X = X; g.ldx = ldx;
            g.C = C; g.ldc = ldc;
            g.beta = make_float2(0.f, 0.f);
            g.gamma = make_float2(0.f, 0.f);
            memcpy(&g.beta, &beta, sizeof(T));
            memcpy(&g.gamma, &minus_one, sizeof(T));
            g.beta_zero = 0;
            g.k_by_col = 0;
            return sp_launch<T>(g, st);
        }
    }
    GemmArgs<T> up;
    up.M = M; up.N = N; up.K = K;
    up.A = A; up.lda = lda;
    up.B = X; up.ldb = ldx;
    up.C = C; up.ldc = ldc;
    up.gamma = minus_one;
    up.beta = beta;
    up.beta_zero = 0; up.a_lower = 0;
    up.b_rowmajor = 1; up.c_rowmajor = 0;
    return gemm_launch<T>(up, st);
}

// Block apply for the single-precision types on the update kernel:
//   X_t^T = gamma * R_t^T * (D_t^{-1})^T,
// with R_t^T the row-major panel P (= a column-major n x mb matrix, ld ldx)
// and (D_t^{-1})^T read as a row-major mb x mb matrix from W_t (column-
// major, ld nb); the result, column-major n x mb with ld ldx, is the
// row-major X_t panel.  (D_t^{-1})^T is upper triangular, so a column tile
// stops its K loop at the tile's last column.  Returns kSpNotApplicable when
// the operands are not 16-byte aligned.
constexpr int kSpNotApplicable = -200000;
template <typename T>
static int apply_sp_launch(int64_t mb, int64_t n, const T *Wt, int64_t nb, const T *P, int64_t ldx, T *Xw, T gamma,
                           cudaStream_t st) {
    if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value) {
        if (((reinterpret_cast<uintptr_t>(Wt) | reinterpret_cast<uintptr_t>(P) | reinterpret_cast<uintptr_t>(Xw)) &
             15) != 0 || (nb * (int64_t)sizeof(T)) % 16 || (ldx * (int64_t)sizeof(T)) % 16)
            return kSpNotApplicable;
        SpArgs g;
        g.M = n; g.N = mb; g.K = mb;
        g.A = P; g.lda = ldx;
        g.X = Wt; g.ldx = nb;
        g.C = Xw; g.ldc = ldx;
        g.beta = make_float2(0.f, 0.f);
        g.gamma = make_float2(0.f, 0.f);
        memcpy(&g.gamma, &gamma, sizeof(T));
        g.beta_zero = 1;
        g.k_by_col = 1;
        return sp_launch<T>(g, st);
    } else {
        (void)mb; (void)n; (void)Wt; (void)nb; (void)P; (void)ldx; (void)Xw; (void)gamma; (void)st;
        return kSpNotApplicable;
    }
}

template <typename T, int IB>
static int invert_diagonal_blocks(const T *L, int64_t lda, int64_t m, int nb, T *W, cudaStream_t st) {
    const int tb = (int)((m + nb - 1) / nb);
    inv_diag_l1_kernel<T, IB><<<tb * 8, IB, 0, st>>>(L, lda, m, nb, W);
    int rc = launch_status();
    if (rc) return rc;
    constexpr size_t smem = inv_offdiag_smem<T, IB>();
    auto kern = inv_offdiag_kernel<T, IB>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_status(e);
    }
    kern<<<dim3(tb, 7), 256, smem, st>>>(L, lda, m, nb, W, 0, 0);
    return launch_status();
}

// f32 and c64: the diagonal blocks of nb = 128, 256 or 512 rows inverted
// level by level.  Every 128-row diagonal block in one CTA
// (inv_block128_kernel), then for s = 128, 256 .. nb/2 the lower-left block
// of every 2s-row diagonal block [[A, 0], [C, D]] -- -D^{-1} (C A^{-1}), the
// same formula as inside the kernel -- by two batched GEMMs, the middle
// product in tmp (at least ceil(m/nb) (nb/2)^2 elements).  The diagonal
// block whose rows run past m (the last one) has its GEMMs cut to its valid
// rows, or its lower-left block zeroed when none are.
template <typename T>
static int invert_blocks_doubling(const T *L, int64_t lda, int64_t m, int nb, T *W, T *tmp, cudaStream_t st) {
    const int64_t tb = (m + nb - 1) / nb;
    constexpr size_t ismem = inv_block128_smem<T>();
    int rc = cuda_status(
        cudaFuncSetAttribute(inv_block128_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ismem));
    if (rc) return rc;
    inv_block128_kernel<T><<<(unsigned)(tb * (nb / kInvN)), 256, ismem, st>>>(L, lda, m, W, nb, nullptr, 0);
    if ((rc = launch_status())) return rc;
    T one, minus_one;
    memset(&one, 0, sizeof(T));
    reinterpret_cast<typename Elem<T>::Real *>(&one)[0] = 1;
    minus_one = one;
    reinterpret_cast<typename Elem<T>::Real *>(&minus_one)[0] = -1;
    const int64_t sW = (int64_t)nb * nb, sL = (int64_t)nb * (lda + 1);
    for (int s = kInvN; s < nb && !rc; s *= 2) {
        for (int o = 0; o < nb && !rc; o += 2 * s) {
            // blocks t < full have all 2s rows inside the matrix
            const int64_t full = m >= o + 2 * s ? std::min<int64_t>(tb, (m - o - 2 * s) / nb + 1) : 0;
            auto run = [&](int64_t t, int64_t count, int64_t rows) {
                // C A^{-1} into tmp (rows x s), then -D^{-1} (C A^{-1}) into W_t
                GemmArgs<T> g1{};
                g1.M = rows, g1.N = s, g1.K = s;
                g1.A = L + (t * nb + o) * (lda + 1) + s, g1.lda = lda, g1.sA = sL;
                g1.B = W + t * sW + (int64_t)o * (nb + 1), g1.ldb = nb, g1.sB = sW;
                g1.C = tmp, g1.ldc = s, g1.sC = (int64_t)s * s;
                g1.gamma = one, g1.beta = one, g1.beta_zero = 1;
                int r = gemm_launch<T>(g1, st, (int)count);
                if (r) return r;
                GemmArgs<T> g2{};
                g2.M = s, g2.N = s, g2.K = rows;
                g2.A = W + t * sW + (int64_t)(o + s) * (nb + 1), g2.lda = nb, g2.sA = sW, g2.a_lower = 1;
                g2.B = tmp, g2.ldb = s, g2.sB = (int64_t)s * s;
                g2.C = W + t * sW + (int64_t)o * nb + o + s, g2.ldc = nb, g2.sC = sW;
                g2.gamma = minus_one, g2.beta = one, g2.beta_zero = 1;
                return gemm_launch<T>(g2, st, (int)count);
            };
            if (full > 0) rc = run(0, full, s);
            if (!rc && full < tb) {
                const int64_t t = tb - 1, rows = m - (t * nb + o + s);
                if (rows > 0)
                    rc = run(t, 1, rows);
                else
                    rc = cuda_status(cudaMemset2DAsync(W + t * sW + (int64_t)o * nb + o + s, nb * sizeof(T), 0,
                                                       s * sizeof(T), s, st));
            }
        }
    }
    return rc;
}

// The few-right-hand-sides path (few_rhs.cuh): n <= kFewMaxN columns of a
// column-major system of order m > kFewMinM, 16-byte aligned L columns, and
// its data (few_rhs_bytes, which blocked_workspace_bytes covers) within the
// workspace of ws_bytes.
constexpr int64_t kFewMinM = 512;

// complex128 only up to four columns: from five on, each block row's FP64
// work on the chain (one SM) outweighs what the kernel saves, and the
// blocked path is faster (m = 16384, n = 8: 37 against 30 ms; n = 3: 19
// against 30 ms).
template <typename T>
static bool few_rhs_usable(int64_t m, int64_t n, const T *L, int64_t lda, size_t ws_bytes) {
    const int64_t max_n = std::is_same<T, double2>::value ? 4 : kFewMaxN;
    return n >= 1 && n <= max_n && m > kFewMinM && ((reinterpret_cast<uintptr_t>(L) & 15) == 0) &&
           (lda * (int64_t)sizeof(T)) % 16 == 0 && few_rhs_bytes((int)sizeof(T), m, n) <= ws_bytes;
}

// The persistent kernel with the right-hand-side count compiled in.  CL:
// clusters of four (else two) consecutive block rows, which hand x_t to the
// next one in shared memory -- the grid a multiple of the cluster, every
// cluster resident (a cooperative launch); kFewNoCluster when neither size
// can be placed.  Without CL a plain cooperative launch.
constexpr int kFewNoCluster = -300000;
template <typename T, bool CL>
static int few_rhs_launch(int64_t n, int64_t tb, void **args, cudaStream_t st) {
    constexpr size_t smem = few_rhs_smem<T, CL>();
    auto kern = n <= 1   ? few_rhs_kernel<T, 1, CL>
                : n <= 2 ? few_rhs_kernel<T, 2, CL>
                : n <= 4 ? few_rhs_kernel<T, 4, CL>
                         : few_rhs_kernel<T, 8, CL>;
    int rc = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    if (rc) return rc;
    if constexpr (CL) {
        for (int K : {4, 2}) {
            cudaLaunchAttribute at[2];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)K;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            at[1].id = cudaLaunchAttributeCooperative;
            at[1].val.cooperative = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)K);
            cfg.blockDim = dim3(320);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
                (void)cudaGetLastError();
                continue;
            }
            const int64_t want = (tb + K - 1) / K;
            cfg.gridDim = dim3((unsigned)((want < clusters ? want : clusters) * K));
            cfg.numAttrs = 2;
            if (cudaLaunchKernelExC(&cfg, (const void *)kern, args) == cudaSuccess) return TRSM_SUCCESS;
            (void)cudaGetLastError();  // e.g. too many blocks for a cooperative launch: the next size
        }
        return kFewNoCluster;
    } else {
        int dev = 0, sms = 0, per_sm = 0;
        rc = cuda_status(cudaGetDevice(&dev));
        if (!rc) rc = cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        if (!rc) rc = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 320, smem));
        if (!rc && per_sm < 1) rc = TRSM_ERR_CUDA_BASE + (int)cudaErrorInvalidConfiguration;
        if (rc) return rc;
        const int64_t cap = (int64_t)sms * per_sm;
        const unsigned grid = (unsigned)(tb < cap ? tb : cap);
        return cuda_status(cudaLaunchCooperativeKernel((const void *)kern, dim3(grid), dim3(320), args, smem, st));
    }
}

// The inversion of the diagonal blocks (few_nb<T>() rows), then the
// persistent kernel (a cooperative launch in clusters: its CTAs wait on one
// another's results, so all of them must be resident at once).  L and the inverted
// blocks are read by TMA tensor copies: float views, a column's block of
// rows as boxes of at most 256 floats.
template <typename T>
static int few_rhs_solve(const T *L, int64_t lda, int64_t m, int64_t n, T *B, int64_t ldb, T alpha, void *ws,
                         cudaStream_t st, float *inv_ms, float *solve_ms) {
    using Cfg = FewCfg<T, false>;  // the geometry (NB, Q, BR, KC) is the same in both forms
    constexpr int64_t NB = Cfg::NB;
    const int64_t tb = (m + NB - 1) / NB;
    T *W = static_cast<T *>(ws);
    T *xpub = reinterpret_cast<T *>(static_cast<char *>(ws) + round256(tb * NB * NB * (int64_t)sizeof(T)));
    CUtensorMap mapL, mapW;
    {
        const uint64_t dl[3] = {(uint64_t)(m * Cfg::Q), (uint64_t)m, 1};
        const uint64_t sl[2] = {(uint64_t)(lda * (int64_t)sizeof(T)), (uint64_t)(lda * (int64_t)sizeof(T) * m)};
        const uint32_t box[3] = {(uint32_t)(Cfg::BR * Cfg::Q), (uint32_t)Cfg::KC, 1};
        int rc = encode_f32_map(&mapL, L, 3, dl, sl, box, false);
        if (rc) return rc;
        const uint64_t dw[3] = {(uint64_t)(NB * Cfg::Q), (uint64_t)(tb * NB), 1};
        const uint64_t sw[2] = {(uint64_t)(NB * (int64_t)sizeof(T)), (uint64_t)(NB * (int64_t)sizeof(T) * tb * NB)};
        rc = encode_f32_map(&mapW, W, 3, dw, sw, box, false);
        if (rc) return rc;
    }
    cudaEvent_t e[3] = {nullptr, nullptr, nullptr};
    if (inv_ms)
        for (auto &x : e) cudaEventCreate(&x);
    if (inv_ms) cudaEventRecord(e[0], st);
    // every word of the published copy of X unset (all ones) until written
    int rc = TRSM_SUCCESS;
    if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value) {
        // one CTA per diagonal block, the whole block in shared memory; it
        // also clears its block row of the published copy
        constexpr size_t ismem = inv_block128_smem<T>();
        static_assert(NB == kInvN, "block rows of 128");
        rc = cuda_status(cudaFuncSetAttribute(inv_block128_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)ismem));
        if (!rc) {
            inv_block128_kernel<T><<<(unsigned)tb, 256, ismem, st>>>(
                L, lda, m, W, (int)NB, reinterpret_cast<uint32_t *>(xpub), n * NB * (int64_t)sizeof(T) / 4);
            rc = launch_status();
        }
    } else {
        rc = invert_diagonal_blocks<T, (int)NB / 8>(L, lda, m, (int)NB, W, st);
        if (!rc) rc = cuda_status(cudaMemsetAsync(xpub, 0xff, (size_t)(tb * n * NB) * sizeof(T), st));
    }
    int *status = nullptr;
    if (!rc) rc = device_status_word(&status);
    if (inv_ms) cudaEventRecord(e[1], st);
    if (!rc) {
        const int ni = (int)n;
        const int64_t limit = int64_t(1) << 22;  // polls of a published block row (each a round trip to L2)
        void *args[] = {(void *)&mapL, (void *)&mapW, (void *)&m, (void *)&ni, (void *)&B, (void *)&ldb,
                        (void *)&alpha, (void *)&xpub, (void *)&status, (void *)&limit};
        // The cluster form for f32 with two or more columns and for complex64
        // (measured faster there); not for one f32 column (0.24 ms without
        // against 0.26 ms with, m = 16384) nor for the FP64 types, whose chain
        // is bound by one SM's FP64 rate.
        rc = kFewNoCluster;
        if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value)
            if (std::is_same<T, float2>::value || n > 1) rc = few_rhs_launch<T, true>(n, tb, args, st);
        if (rc == kFewNoCluster) rc = few_rhs_launch<T, false>(n, tb, args, st);
    }
    if (inv_ms) {
        cudaEventRecord(e[2], st);
        cudaEventSynchronize(e[2]);
        cudaEventElapsedTime(inv_ms, e[0], e[1]);
        cudaEventElapsedTime(solve_ms, e[1], e[2]);
        for (auto &x : e) cudaEventDestroy(x);
    }
    return rc;
}

struct PhaseTimer {
    bool on = false;
    cudaStream_t st = nullptr;
    cudaEvent_t ev[2] = {nullptr, nullptr};
    float acc[3] = {0, 0, 0};
    int open(cudaStream_t s) {
        on = true;
        st = s;
        for (auto &e : ev)
            if (cudaEventCreate(&e) != cudaSuccess) return launch_status();
        return TRSM_SUCCESS;
    }
    void begin() {
        if (on) cudaEventRecord(ev[0], st);
    }
    int end(int phase) {
        if (!on) return TRSM_SUCCESS;
        cudaEventRecord(ev[1], st);
        cudaError_t e = cudaEventSynchronize(ev[1]);
        if (e != cudaSuccess) return cuda_status(e);
        float ms = 0;
        cudaEventElapsedTime(&ms, ev[0], ev[1]);
        acc[phase] += ms;
        return TRSM_SUCCESS;
    }
    ~PhaseTimer() {
        for (auto &e : ev)
            if (e) cudaEventDestroy(e);
    }
};

template <typename T> constexpr int elem_code();
template <> constexpr int elem_code<float>() { return 0; }
template <> constexpr int elem_code<double>() { return 1; }
template <> constexpr int elem_code<float2>() { return 2; }
template <> constexpr int elem_code<double2>() { return 3; }

template <typename T>
int blocked_solve_typed(const BlockedArgs &a, cudaStream_t st) {
    const int64_t m = a.m, n = a.n, nb = a.nb;
    const T *L = static_cast<const T *>(a.A);
    T *B = static_cast<T *>(a.B);
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    const int64_t tbk = (m + nb - 1) / nb;
    const int64_t ldx = panel_ld(n);
    T *W = static_cast<T *>(a.ws);
    T *Xw = reinterpret_cast<T *>(static_cast<char *>(a.ws) + round256(tbk * nb * nb * (int64_t)sizeof(T)));
    T *Pw = reinterpret_cast<T *>(reinterpret_cast<char *>(Xw) + round256(nb * ldx * (int64_t)sizeof(T)));
    void *tc_panels = nullptr;
    if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value)
        tc_panels = reinterpret_cast<char *>(Pw) + round256(nb * ldx * (int64_t)sizeof(T));

    if (!a.tri_rhs && (a.nb_from_table || nb == few_nb<T>()) &&
        few_rhs_usable<T>(m, n, L, a.lda, blocked_workspace_bytes(elem_code<T>(), m, n, nb))) {
        // a handful of columns: the persistent few-RHS kernel (profile: the
        // inversion in ms[0], the solve in ms[2])
        if (a.ms) a.ms[1] = 0.f;
        T alpha0;
        memcpy(&alpha0, a.alpha, sizeof(T));
        return few_rhs_solve<T>(L, a.lda, m, n, B, a.ldb, alpha0, a.ws, st, a.ms ? &a.ms[0] : nullptr,
                                a.ms ? &a.ms[2] : nullptr);
    }

    PhaseTimer timer;
    int rc = TRSM_SUCCESS;
    if (a.ms && (rc = timer.open(st))) return rc;

    // Phase 0: invert every diagonal block D_t (independent, one CTA each).
    timer.begin();
    if (nb != 128 && nb != 256 && nb != 512) return -9;
    if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value) {
        // the middle products live in the tensor-core panels, unused until the solve
        rc = invert_blocks_doubling<T>(L, a.lda, m, (int)nb, W, static_cast<T *>(tc_panels), st);
    } else {
        switch (nb) {
            case 128: rc = invert_diagonal_blocks<T, 16>(L, a.lda, m, (int)nb, W, st); break;
            case 256: rc = invert_diagonal_blocks<T, 32>(L, a.lda, m, (int)nb, W, st); break;
            default: rc = invert_diagonal_blocks<T, 64>(L, a.lda, m, (int)nb, W, st); break;
        }
    }
    if (rc || (rc = timer.end(0))) return rc;

    T one;
    memset(&one, 0, sizeof(T));
    reinterpret_cast<typename Elem<T>::Real *>(&one)[0] = 1;
    T minus_one = one;
    reinterpret_cast<typename Elem<T>::Real *>(&minus_one)[0] = -1;

    const int64_t tb = (m + nb - 1) / nb;
    if constexpr (std::is_same<T, float>::value) {
        if (tc_panels && tc_fused_usable(m, n, nb)) {
            // look-ahead form (tc_gemm.cu): every launch but the last is an
            // update with the previous block's apply folded in (phase 2);
            // the last holds the two remaining applies (phase 1)
            timer.begin();
            TcSide *side = nullptr;
            rc = tc_side_acquire(st, &side);
            if (!rc) rc = tc_fused_prepare_side(m, n, nb, L, a.lda, W, B, a.ldb, tc_panels, st, side, a.tri_rhs);
            for (int64_t t = 0; !rc && t + 1 < tb; ++t)
                rc = tc_fused_step_side(t, m, n, nb, L, a.lda, W, B, a.ldb, alpha, tc_panels, st, side, a.tri_rhs);
            tc_side_release(side);
            if (rc || (rc = timer.end(2))) return rc;
            timer.begin();
            rc = tc_fused_step(tb - 1, m, n, nb, L, a.lda, W, B, a.ldb, alpha, tc_panels, st, a.tri_rhs);
            if (rc || (rc = timer.end(1))) return rc;
            if (a.ms)
                for (int q = 0; q < 3; ++q) a.ms[q] = timer.acc[q];
            return TRSM_SUCCESS;
        }
    }
    if constexpr (std::is_same<T, float2>::value) {
        if (tc_panels && tc_fused_usable_c64(m, n, nb)) {
            // the look-ahead form in real form (tc_gemm.cu), phases as for f32
            timer.begin();
            rc = tc_fused_prepare_c64(m, n, nb, L, a.lda, W, B, a.ldb, tc_panels, st, a.tri_rhs);
            for (int64_t t = 0; !rc && t + 1 < tb; ++t)
                rc = tc_fused_step_c64(t, m, n, nb, L, a.lda, W, B, a.ldb, alpha, tc_panels, st, a.tri_rhs);
            if (rc || (rc = timer.end(2))) return rc;
            timer.begin();
            rc = tc_fused_step_c64(tb - 1, m, n, nb, L, a.lda, W, B, a.ldb, alpha, tc_panels, st, a.tri_rhs);
            if (rc || (rc = timer.end(1))) return rc;
            if (a.ms)
                for (int q = 0; q < 3; ++q) a.ms[q] = timer.acc[q];
            return TRSM_SUCCESS;
        }
    }
    for (int64_t t = 0; t < tb; ++t) {
        const int64_t r0 = t * nb;
        const int64_t mb = (m - r0 < nb) ? m - r0 : nb;
        // a lower-triangular right-hand side (the identity of the triangular
        // inverse) has no nonzero column past block t in block rows <= t, so
        // X_t and this step's update touch only the first (t+1) nb columns
        const int64_t nt = (a.tri_rhs && (t + 1) * nb < n) ? (t + 1) * nb : n;
        // Phase 1: X_t = gamma * D_t^{-1} R_t into the panel (gamma = alpha at
        // t = 0; later block rows already carry alpha through the updates).
        const T gamma = (t == 0) ? alpha : one;
        if constexpr (std::is_same<T, float>::value) {
            // both products on the tensor cores: X_t straight over R_t in B,
            // its split copy straight into the update's operand panels
            const bool has_update = r0 + nb < m;
            if (tc_panels && tc_apply_usable(mb, nt) &&
                (!has_update || tc_update_usable(m - r0 - nb, nt, nb))) {
                timer.begin();
                rc = tc_apply_f32(mb, nt, W + t * nb * nb, nb, B + r0, a.ldb, gamma, m, tc_panels, has_update, st);
                if (rc || (rc = timer.end(1))) return rc;
                timer.begin();
                if (has_update) {
                    const T beta = (t == 0) ? alpha : one;
                    rc = tc_update_f32(m - r0 - nb, nt, nb, L + r0 * a.lda + r0 + nb, a.lda, nullptr, 0, B + r0 + nb,
                                       a.ldb, beta, m, tc_panels, st);
                    if (rc) return rc;
                }
                if ((rc = timer.end(2))) return rc;
                continue;
            }
        }
        if constexpr (std::is_same<T, float2>::value) {
            // the same with the complex products in real form
            const bool has_update = r0 + nb < m;
            if (tc_panels && tc_apply_usable_c64(mb, nt) &&
                (!has_update || tc_update_usable(m - r0 - nb, 2 * nt, 2 * nb))) {
                timer.begin();
                rc = tc_apply_c64(mb, nt, W + t * nb * nb, nb, B + r0, a.ldb, gamma, m, tc_panels, has_update, st);
                if (rc || (rc = timer.end(1))) return rc;
                timer.begin();
                if (has_update) {
                    const T beta = (t == 0) ? alpha : one;
                    rc = tc_update_c64(m - r0 - nb, nt, nb, L + r0 * a.lda + r0 + nb, a.lda, nullptr, 0, B + r0 + nb,
                                       a.ldb, beta, m, tc_panels, st);
                    if (rc) return rc;
                }
                if ((rc = timer.end(2))) return rc;
                continue;
            }
        }
        timer.begin();
        rc = kSpNotApplicable;
        if constexpr (std::is_same<T, float>::value || std::is_same<T, float2>::value) {
            // R_t (column-major block row of B) -> row-major panel P
            const dim3 tgrid((unsigned)((mb + 31) / 32), (unsigned)((nt + 31) / 32));
            transpose_kernel<T><<<tgrid, dim3(32, 8), 0, st>>>(B + r0, a.ldb, Pw, ldx, nt, mb);
            if ((rc = launch_status())) return rc;
            rc = apply_sp_launch<T>(mb, nt, W + t * nb * nb, nb, Pw, ldx, Xw, gamma, st);
        }
        if (rc == kSpNotApplicable) {
            GemmArgs<T> ap;
            ap.M = mb; ap.N = nt; ap.K = mb;
            ap.A = W + t * nb * nb; ap.lda = nb;
            ap.B = B + r0; ap.ldb = a.ldb;
            ap.C = Xw; ap.ldc = ldx;
            ap.gamma = gamma;
            ap.beta = one; ap.beta_zero = 1; ap.a_lower = 1;
            ap.b_rowmajor = 0; ap.c_rowmajor = 1;
            rc = gemm_launch<T>(ap, st);
        }
        if (rc) return rc;
        if ((rc = timer.end(1))) return rc;

        // Phase 2: trailing update  B[r0+nb:, :] = beta*B[...] - L[r0+nb:, r0:r0+nb] X_t
        // (beta = alpha at t = 0: the first touch of every later block row),
        // and X_t back into its block row of B.
        timer.begin();
        if (r0 + nb < m) {
            const T beta = (t == 0) ? alpha : one;
            const T *Lp = L + r0 * a.lda + r0 + nb;
            if ((rc = update_launch<T>(m - r0 - nb, nt, nb, Lp, a.lda, Xw, ldx, B + r0 + nb, a.ldb, beta,
                                       minus_one, st, m, tc_panels)))
                return rc;
        }
        {
            // X_t (row-major panel) back into its block row of B (column-major)
            const dim3 grid((unsigned)((nt + 31) / 32), (unsigned)((mb + 31) / 32));
            transpose_kernel<T><<<grid, dim3(32, 8), 0, st>>>(Xw, ldx, B + r0, a.ldb, mb, nt);
            if ((rc = launch_status())) return rc;
        }
        if ((rc = timer.end(2))) return rc;
    }
    if (a.ms)
        for (int q = 0; q < 3; ++q) a.ms[q] = timer.acc[q];
    return TRSM_SUCCESS;
}

// ---------------------------------------------------------------------------
// The blocked path over a strided batch of column-major systems in one
// sequence of launches: every kernel carries the system index in its grid's
// last dimension (llama.cpp PR 17457 leaves its 128 x 128 batched case
// unsupported; one launch sequence serves any batch here).  The inversion
// runs once per distinct A (once in all when the systems share A, sA == 0);
// then per block row t one apply X_t = gamma D_t^{-1} R_t, one trailing
// update and one copy of X_t back into B, each over the whole batch.  The
// products run on the FMA-pipe kernels (these systems are too small for
// the tensor-core tiles).  Workspace (256-byte aligned): the inverted blocks
// (cnt or 1 systems x ceil(m/nb) x nb x nb), then the X_t and R_t panels
// (cnt x nb x panel_ld(n) each).
// ---------------------------------------------------------------------------
template <typename T>
int blocked_solve_batched_typed(const BatchedBlockedArgs &a, cudaStream_t st) {
    const int64_t m = a.m, n = a.n, nb = a.nb, cnt = a.batch;
    if (cnt <= 0) return TRSM_SUCCESS;
    if (cnt > 65535) return -12;
    const bool shared_a = a.strideA == 0;
    const T *L = static_cast<const T *>(a.A);
    T *B = static_cast<T *>(a.B);
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    const int64_t tb = (m + nb - 1) / nb;
    const int64_t ldx = panel_ld(n);
    const int64_t sW = shared_a ? 0 : tb * nb * nb;  // element stride of the systems' inverted blocks
    const int64_t sX = nb * ldx;
    const int nA = shared_a ? 1 : (int)cnt;
    T *W = static_cast<T *>(a.ws);
    T *Xw = reinterpret_cast<T *>(static_cast<char *>(a.ws) + round256((int64_t)nA * tb * nb * nb * sizeof(T)));
    T *Pw = reinterpret_cast<T *>(reinterpret_cast<char *>(Xw) + round256(cnt * sX * (int64_t)sizeof(T)));
    const int nz = (int)cnt;
    int rc = TRSM_SUCCESS;

    // Phase 0: every diagonal block of every distinct A
    auto invert = [&](auto ib_tag) -> int {
        constexpr int IB = decltype(ib_tag)::value;
        inv_diag_l1_kernel<T, IB><<<dim3((unsigned)(tb * 8), (unsigned)nA), IB, 0, st>>>(L, a.lda, m, (int)nb, W,
                                                                                      a.strideA, sW);
        int r = launch_status();
        if (r) return r;
        constexpr size_t smem = inv_offdiag_smem<T, IB>();
        auto kern = inv_offdiag_kernel<T, IB>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return cuda_status(e);
        }
        kern<<<dim3((unsigned)tb, 7, (unsigned)nA), 256, smem, st>>>(L, a.lda, m, (int)nb, W, a.strideA, sW);
        return launch_status();
    };
    switch (nb) {
        case 128: rc = invert(std::integral_constant<int, 16>{}); break;
        case 256: rc = invert(std::integral_constant<int, 32>{}); break;
        case 512: rc = invert(std::integral_constant<int, 64>{}); break;
        default: return -9;
    }
    if (rc) return rc;

    T one;
    memset(&one, 0, sizeof(T));
    reinterpret_cast<typename Elem<T>::Real *>(&one)[0] = 1;
    T minus_one = one;
    reinterpret_cast<typename Elem<T>::Real *>(&minus_one)[0] = -1;
    constexpr bool kSp = std::is_same<T, float>::value || std::is_same<T, float2>::value;
    const int64_t eb = (int64_t)sizeof(T);
    // the FMA-pipe single-precision kernels read A in 16-byte chunks
    const bool sp_ok = kSp && ((reinterpret_cast<uintptr_t>(L) & 15) == 0) && (a.lda * eb) % 16 == 0 &&
                       (a.strideA * eb) % 16 == 0;

    for (int64_t t = 0; t < tb; ++t) {
        const int64_t r0 = t * nb;
        const int64_t mb = (m - r0 < nb) ? m - r0 : nb;
        const T gamma = (t == 0) ? alpha : one;
        const T *Wt = W + t * nb * nb;
        // Phase 1: X_t = gamma D_t^{-1} R_t into the row-major panels
        rc = kSpNotApplicable;
        if constexpr (kSp) {
            const dim3 tgrid((unsigned)((mb + 31) / 32), (unsigned)((n + 31) / 32), (unsigned)nz);
            transpose_kernel<T><<<tgrid, dim3(32, 8), 0, st>>>(B + r0, a.ldb, Pw, ldx, n, mb, a.strideB, sX);
            if ((rc = launch_status())) return rc;
            SpArgs g;
            g.M = n; g.N = mb; g.K = mb;
            g.A = Pw; g.lda = ldx; g.sA = sX;
            g.X = Wt; g.ldx = nb; g.sX = sW;
            g.C = Xw; g.ldc = ldx; g.sC = sX;
            g.beta = make_float2(0.f, 0.f);
            g.gamma = make_float2(0.f, 0.f);
            memcpy(&g.gamma, &gamma, sizeof(T));
            g.beta_zero = 1;
            g.k_by_col = 1;
            rc = sp_launch<T>(g, st, nz);
        }
        if (rc == kSpNotApplicable) {
            GemmArgs<T> ap;
            ap.M = mb; ap.N = n; ap.K = mb;
            ap.A = Wt; ap.lda = nb; ap.sA = sW;
            ap.B = B + r0; ap.ldb = a.ldb; ap.sB = a.strideB;
            ap.C = Xw; ap.ldc = ldx; ap.sC = sX;
            ap.gamma = gamma;
            ap.beta = one; ap.beta_zero = 1; ap.a_lower = 1;
            ap.b_rowmajor = 0; ap.c_rowmajor = 1;
            rc = gemm_launch<T>(ap, st, nz);
        }
        if (rc) return rc;
        // Phase 2: B[r0+nb:, :] = beta B[...] - L[r0+nb:, t-block] X_t
        if (r0 + nb < m) {
            const T beta = (t == 0) ? alpha : one;
            const T *Lp = L + r0 * a.lda + r0 + nb;
            rc = kSpNotApplicable;
            if constexpr (kSp) {
                if (sp_ok && ((reinterpret_cast<uintptr_t>(Lp) & 15) == 0)) {
                    SpArgs g;
                    g.M = m - r0 - nb; g.N = n; g.K = nb;
                    g.A = Lp; g.lda = a.lda; g.sA = a.strideA;
                    g.X = Xw; g.ldx = ldx; g.sX = sX;
                    g.C = B + r0 + nb; g.ldc = a.ldb; g.sC = a.strideB;
                    g.beta = make_float2(0.f, 0.f);
                    g.gamma = make_float2(0.f, 0.f);
                    memcpy(&g.beta, &beta, sizeof(T));
                    memcpy(&g.gamma, &minus_one, sizeof(T));
                    g.beta_zero = 0;
                    g.k_by_col = 0;
                    rc = sp_launch<T>(g, st, nz);
                }
            }
            if (rc == kSpNotApplicable) {
                GemmArgs<T> up;
                up.M = m - r0 - nb; up.N = n; up.K = nb;
                up.A = Lp; up.lda = a.lda; up.sA = a.strideA;
                up.B = Xw; up.ldb = ldx; up.sB = sX;
                up.C = B + r0 + nb; up.ldc = a.ldb; up.sC = a.strideB;
                up.gamma = minus_one;
                up.beta = beta;
                up.beta_zero = 0; up.a_lower = 0;
                up.b_rowmajor = 1; up.c_rowmajor = 0;
                rc = gemm_launch<T>(up, st, nz);
            }
            if (rc) return rc;
        }
        // X_t (row-major panels) back into the block rows of B
        const dim3 grid((unsigned)((n + 31) / 32), (unsigned)((mb + 31) / 32), (unsigned)nz);
        transpose_kernel<T><<<grid, dim3(32, 8), 0, st>>>(Xw, ldx, B + r0, a.ldb, mb, n, sX, a.strideB);
        if ((rc = launch_status())) return rc;
    }
    return TRSM_SUCCESS;
}

}  // namespace trsm
