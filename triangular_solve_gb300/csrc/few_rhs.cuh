// Few right-hand sides (n <= 8) on one large system.
//
// With a handful of columns the blocked path's GEMMs have no width: every
// product is a thin matrix-vector product bound by reading L once from HBM,
// and the per-block-row launches dominate.  This path keeps the blocked
// algorithm of "Hierarchical Shared Memory-Aware Optimization for TRSM on GPU
// Platforms" -- the diagonal blocks inverted up front (W_t = D_t^{-1}, the
// same inversion kernels), then per block row t
//     x_t = W_t (alpha b_t - sum_{s<t} L_ts x_s)
// -- but runs all block rows in one cooperatively launched persistent
// kernel.  The CTA that owns block row t streams its tiles L_ts (s < t) and
// then W_t through a ring of cp.async stages, independently of the solve, so
// every tile is on chip before it is needed; it folds tile s in as soon as
// the owner of block row s has published x_s (a flag per block row, waits
// bounded), and publishes x_t in turn.  The reduction sum_{s<t} L_ts x_s is
// therefore spread over the owners of the block rows below, in parallel,
// and only one 128 x 128 product and the application of W_t per block row
// lie on the dependency chain.
#pragma once

#include "common.cuh"
#include "gemm_sp.cuh"  // cp_async16_zfill
#include "mbarrier.cuh"  // record_timeout

namespace trsm {

constexpr int kFewNB = 128;   // block rows of the few-RHS path
constexpr int kFewMaxN = 8;   // right-hand sides it takes

template <typename T>
struct FewCfg {
    static constexpr int KC = 32;                                  // columns of a streamed chunk
    static constexpr int kChunk = kFewNB * KC;                     // elements
    static constexpr int ST = sizeof(T) >= 16 ? 3 : 4;             // ring stages
    static constexpr int VE = 16 / (int)sizeof(T) > 0 ? 16 / (int)sizeof(T) : 1;  // elements per 16 bytes
    static constexpr size_t kSmem =
        (size_t)ST * kChunk * sizeof(T) + 2 * (size_t)kFewNB * kFewMaxN * sizeof(T);
};

__device__ __forceinline__ float add2_(float a, float b) { return a + b; }
__device__ __forceinline__ double add2_(double a, double b) { return a + b; }
__device__ __forceinline__ float2 add2_(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ double2 add2_(double2 a, double2 b) { return make_double2(a.x + b.x, a.y + b.y); }

__device__ __forceinline__ int ld_acquire_flag(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_flag(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

// 256 threads: thread (row, half) = (tid % 128, tid / 128); a chunk's KC
// columns are split between the two halves, whose partial sums meet in
// shared memory at the end of each block row.
// NC: right-hand sides the registers and loops are sized for (n <= NC; the
// launcher picks the smallest of 1, 2, 4, 8): a guarded loop over a fixed
// eight would still issue the idle columns' FMAs, which on the FP64 pipe
// cost as much as the real ones.
template <typename T, int NC>
__global__ void __launch_bounds__(256, 1)
    few_rhs_kernel(const T *__restrict__ L, int64_t lda, int64_t m, int n, T *B, int64_t ldb,
                   const T *__restrict__ W, const T alpha, int *flags, int *status, const int64_t wait_limit) {
    using C = FewCfg<T>;
    constexpr int NB = kFewNB, KC = C::KC, ST = C::ST, VE = C::VE, KPT = NB / KC;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *ring = reinterpret_cast<T *>(smem_raw);  // [ST][KC][NB], column j of a chunk at j*NB
    T *xs = ring + ST * C::kChunk;              // [NB][kFewMaxN]: x_s of the current tile, or r_t
    T *part = xs + NB * kFewMaxN;               // [NB][kFewMaxN]: the second half's partial sums
    __shared__ int abort_flag;
    const int tid = threadIdx.x, row = tid % NB, half = tid / NB;
    const int64_t tb = (m + NB - 1) / NB;
    if (tid == 0) abort_flag = 0;
    __syncthreads();

    for (int64_t t = blockIdx.x; t < tb; t += gridDim.x) {
        const int64_t r0 = t * NB;
        const int64_t nchunks = (t + 1) * KPT;  // tiles s < t of L, then W_t
        // chunk c: columns k0..k0+KC of tile c / KPT, rows r0..r0+NB (zero past m)
        auto issue = [&](int64_t c) {
            const int64_t s = c / KPT;
            const int k0 = (int)(c % KPT) * KC;
            T *dst = ring + (c % ST) * C::kChunk;
            const T *src;
            int64_t ld;
            int64_t rows_valid;
            if (s < t) {
                src = L + (s * NB + k0) * lda + r0;
                ld = lda;
                rows_valid = m - r0;
            } else {
                src = W + t * NB * NB + (int64_t)k0 * NB;
                ld = NB;
                rows_valid = NB;
            }
            constexpr int kVecs = KC * NB / VE;
            for (int e = tid; e < kVecs; e += 256) {
                const int j = e / (NB / VE), i0 = (e % (NB / VE)) * VE;
                int bytes = 0;
                if (i0 < rows_valid) bytes = (int)((rows_valid - i0 < VE ? rows_valid - i0 : VE) * sizeof(T));
                cp_async16_zfill(dst + j * NB + i0, bytes ? src + j * ld + i0 : src, bytes);
            }
        };
        for (int c = 0; c < ST - 1; ++c) {
            if (c < nchunks) issue(c);
            cp_async_commit();
        }
        T acc[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c] = zero_of<T>();

        for (int64_t c = 0; c < nchunks; ++c) {
            const int64_t s = c / KPT;
            if (c % KPT == 0) {
                if (s < t) {
                    // x_s, once its owner has published it
                    if (tid == 0) {
                        int64_t spins = 0;
                        while (ld_acquire_flag(flags + s) == 0) {
                            if (++spins > wait_limit) {
                                record_timeout(status);
                                abort_flag = 1;
                                break;
                            }
                            __nanosleep(64);
                        }
                    }
                    __syncthreads();
                    if (abort_flag) {
                        cp_async_wait_all();
                        return;
                    }
                    for (int e = tid; e < NB * NC; e += 256) {
                        const int i = e / NC, cc = e % NC;
                        xs[i * kFewMaxN + cc] = cc < n ? __ldcg(B + cc * ldb + s * NB + i) : zero_of<T>();
                    }
                } else {
                    // every tile is in: r_t = alpha b_t - sum_s L_ts x_s
                    if (half == 1) {
#pragma unroll
                        for (int cc = 0; cc < NC; ++cc)
                            if (cc < n) part[row * kFewMaxN + cc] = acc[cc];
                    }
                    __syncthreads();
                    if (half == 0) {
#pragma unroll
                        for (int cc = 0; cc < NC; ++cc) {
                            if (cc >= n) continue;
                            const T b = (r0 + row < m) ? B[cc * ldb + r0 + row] : zero_of<T>();
                            xs[row * kFewMaxN + cc] = sub_(sub_(mul(alpha, b), acc[cc]), part[row * kFewMaxN + cc]);
                        }
#pragma unroll
                        for (int cc = 0; cc < NC; ++cc)
                            if (cc >= n) xs[row * kFewMaxN + cc] = zero_of<T>();
                    }
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc) acc[cc] = zero_of<T>();
                }
            }
            cp_async_wait<ST - 2>();
            __syncthreads();
            if (c + ST - 1 < nchunks) issue(c + ST - 1);
            cp_async_commit();
            const T *ch = ring + (c % ST) * C::kChunk;
            const int k0 = (int)(c % KPT) * KC;
            // two partial sums per column (even / odd j): independent FMA chains
            T acc2[NC];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) acc2[cc] = zero_of<T>();
#pragma unroll 4
            for (int jj = 0; jj < KC / 2; jj += 2) {
                const int j = half * (KC / 2) + jj;
                const T a0 = ch[j * NB + row], a1 = ch[(j + 1) * NB + row];
                const T *xk = xs + (k0 + j) * kFewMaxN;
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    acc[cc] = fma_(a0, xk[cc], acc[cc]);
                    acc2[cc] = fma_(a1, xk[kFewMaxN + cc], acc2[cc]);
                }
            }
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) acc[cc] = add2_(acc[cc], acc2[cc]);
        }
        // x_t = W_t r_t: the halves meet, X goes over b_t, then the flag
        __syncthreads();
        if (half == 1) {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc)
                if (cc < n) part[row * kFewMaxN + cc] = acc[cc];
        }
        __syncthreads();
        if (half == 0 && r0 + row < m) {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                if (cc >= n) continue;
                const T p = part[row * kFewMaxN + cc];
                B[cc * ldb + r0 + row] = fma_(one_of<T>(), p, acc[cc]);
            }
            __threadfence();  // x_t visible GPU-wide before the flag
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            st_release_flag(flags + t, 1);
        }
    }
    cp_async_wait_all();
}

template <typename T>
constexpr size_t few_rhs_smem() {
    return FewCfg<T>::kSmem;
}

}  // namespace trsm
