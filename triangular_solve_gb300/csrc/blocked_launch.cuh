// Host driver of the blocked path for one element type.
#pragma once

#include "blocked_kernels.cuh"
#include "internal.h"

namespace trsm {

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Workspace: W (T_blocks x NB x NB inverted diagonal blocks) then an NB x n
// panel for X_t, each 256-byte aligned.
inline void blocked_ws_layout(int elem, int64_t m, int64_t n, int64_t nb, int64_t *w_bytes, int64_t *x_bytes) {
    const int64_t tb = (m + nb - 1) / nb;
    *w_bytes = round_up(tb * nb * nb * elem, 256);
    *x_bytes = round_up(nb * (n > 0 ? n : 1) * elem, 256);
}

template <typename T>
static int gemm_launch(const GemmArgs<T> &g, cudaStream_t st) {
    using C = GemmCfg<T>;
    if (g.M <= 0 || g.N <= 0) return TRSM_SUCCESS;
    const dim3 grid((unsigned)((g.M + C::BM - 1) / C::BM), (unsigned)((g.N + C::BN - 1) / C::BN));
    gemm_kernel<T><<<grid, 256, 0, st>>>(g);
    return launch_status();
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
    for (int d = 1; d < 8; ++d) {
        kern<<<dim3(tb, 8 - d), 256, smem, st>>>(L, lda, m, nb, W, d);
        rc = launch_status();
        if (rc) return rc;
    }
    return TRSM_SUCCESS;
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

template <typename T>
int blocked_solve_typed(const BlockedArgs &a, cudaStream_t st) {
    const int64_t m = a.m, n = a.n, nb = a.nb;
    const T *L = static_cast<const T *>(a.A);
    T *B = static_cast<T *>(a.B);
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    int64_t wb, xb;
    blocked_ws_layout((int)sizeof(T), m, n, nb, &wb, &xb);
    T *W = static_cast<T *>(a.ws);
    T *Xw = reinterpret_cast<T *>(static_cast<char *>(a.ws) + wb);

    PhaseTimer timer;
    int rc = TRSM_SUCCESS;
    if (a.ms && (rc = timer.open(st))) return rc;

    // Phase 0: invert every diagonal block D_t (independent, one CTA each).
    timer.begin();
    switch (nb) {
        case 128: rc = invert_diagonal_blocks<T, 16>(L, a.lda, m, (int)nb, W, st); break;
        case 256: rc = invert_diagonal_blocks<T, 32>(L, a.lda, m, (int)nb, W, st); break;
        case 512: rc = invert_diagonal_blocks<T, 64>(L, a.lda, m, (int)nb, W, st); break;
        default: return -9;
    }
    if (rc || (rc = timer.end(0))) return rc;

    T one;
    memset(&one, 0, sizeof(T));
    reinterpret_cast<typename Elem<T>::Real *>(&one)[0] = 1;
    T minus_one = one;
    reinterpret_cast<typename Elem<T>::Real *>(&minus_one)[0] = -1;

    const int64_t tb = (m + nb - 1) / nb;
    for (int64_t t = 0; t < tb; ++t) {
        const int64_t r0 = t * nb;
        const int64_t mb = (m - r0 < nb) ? m - r0 : nb;
        // Phase 1: X_t = gamma * D_t^{-1} R_t into the panel (gamma = alpha at
        // t = 0; later block rows already carry alpha through the updates).
        GemmArgs<T> ap;
        ap.M = mb; ap.N = n; ap.K = mb;
        ap.A = W + t * nb * nb; ap.lda = nb;
        ap.B = B + r0; ap.ldb = a.ldb;
        ap.C = Xw; ap.ldc = nb;
        ap.gamma = (t == 0) ? alpha : one;
        ap.beta = one; ap.beta_zero = 1; ap.a_lower = 1;
        timer.begin();
        if ((rc = gemm_launch<T>(ap, st))) return rc;
        if ((rc = timer.end(1))) return rc;

        // Phase 2: trailing update  B[r0+nb:, :] = beta*B[...] - L[r0+nb:, r0:r0+nb] X_t
        // (beta = alpha at t = 0: the first touch of every later block row),
        // and X_t back into its block row of B.
        timer.begin();
        if (r0 + nb < m) {
            GemmArgs<T> up;
            up.M = m - r0 - nb; up.N = n; up.K = nb;
            up.A = L + r0 * a.lda + r0 + nb; up.lda = a.lda;
            up.B = Xw; up.ldb = nb;
            up.C = B + r0 + nb; up.ldc = a.ldb;
            up.gamma = minus_one;
            up.beta = (t == 0) ? alpha : one;
            up.beta_zero = 0; up.a_lower = 0;
            if ((rc = gemm_launch<T>(up, st))) return rc;
        }
        {
            const int64_t total = mb * n;
            int64_t blocks = (total + 255) / 256;
            if (blocks > 152 * 8) blocks = 152 * 8;
            copy_block_kernel<T><<<(unsigned)blocks, 256, 0, st>>>(Xw, nb, B + r0, a.ldb, mb, n);
            if ((rc = launch_status())) return rc;
        }
        if ((rc = timer.end(2))) return rc;
    }
    if (a.ms)
        for (int q = 0; q < 3; ++q) a.ms[q] = timer.acc[q];
    return TRSM_SUCCESS;
}

}  // namespace trsm
