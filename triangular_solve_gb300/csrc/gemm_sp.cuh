// Trailing-update GEMM for the single-precision types (f32, complex64):
//     C = beta * C + gamma * A * X      (update: gamma = -1)
// A: M x K column-major (the L panel under the diagonal block), X: K x N
// row-major (the X_t panel), C: M x N column-major (the block rows of B
// below the panel).  This contraction is the dominant cost of the blocked
// path ("Hierarchical Shared Memory-Aware Optimization for TRSM on GPU
// Platforms", Table 3: 54.8% of the run at m = 2048 rising to 88.0% at
// m = 8192).
//
// SIMT FFMA kernel: 256 threads as 2 x 4 warps; a lane owns RM x RN
// elements laid out as 16-byte chunks spaced so that every fragment load
// is one conflict-free LDS.128 wavefront (8 distinct A chunks, 4 distinct X
// chunks per warp instruction).  Global tiles arrive through a STAGES-deep
// ring of 16-byte cp.async copies (zero-filled at the edges).
#pragma once

#include "common.cuh"

namespace trsm {

// Per-thread tiles.  The large tiles (CTA 128 x 128 for f32, 128 x 64 for
// complex64) are used when they give at least two waves of CTAs; smaller
// problems (the last block rows, and m of a few thousand) take the SMALL
// tiles (64 x 64 / 64 x 32) so that every SM gets work.
template <typename E, bool SMALL> struct SpCfg;
template <> struct SpCfg<float, false> {
    static constexpr int VE = 4;            // elements per 16-byte chunk
    static constexpr int RM = 8, RN = 8;    // per-thread tile
    static constexpr int BK = 16, STAGES = 4;
};
template <> struct SpCfg<float, true> {
    static constexpr int VE = 4;
    static constexpr int RM = 4, RN = 4;
    static constexpr int BK = 16, STAGES = 4;
};
template <> struct SpCfg<float2, false> {
    static constexpr int VE = 2;
    static constexpr int RM = 8, RN = 4;
    static constexpr int BK = 16, STAGES = 3;
};
template <> struct SpCfg<float2, true> {
    static constexpr int VE = 2;
    static constexpr int RM = 4, RN = 2;
    static constexpr int BK = 16, STAGES = 4;
};

template <typename E, bool SMALL = false>
struct SpTile {
    using C = SpCfg<E, SMALL>;
    static constexpr int VE = C::VE, RM = C::RM, RN = C::RN, BK = C::BK, STAGES = C::STAGES;
    static constexpr int WM = 8 * RM, WN = 4 * RN;   // warp tile (lanes 8 x 4)
    static constexpr int BM = 2 * WM, BN = 4 * WN;   // CTA tile (warps 2 x 4)
    static constexpr int A_STAGE = BK * BM, X_STAGE = BK * BN;  // elements
    static constexpr size_t SMEM = (size_t)STAGES * (A_STAGE + X_STAGE) * sizeof(E);
};

struct SpArgs {
    int64_t M, N, K;
    const void *A;
    int64_t lda;
    const void *X;
    int64_t ldx;
    void *C;
    int64_t ldc;
    float2 beta, gamma;  // C = beta*C + gamma*A*X (.x only for real)
    int beta_zero;       // do not read C
    int k_by_col;        // X(k, c) = 0 for k > c: column tile [n0, n0+BN) stops K at n0 + BN
    int64_t sA = 0, sX = 0, sC = 0;  // grid z: systems of a batch, element strides
};

// 16-byte copy of src_bytes (0..16) with zero fill of the rest.
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ float beta_of(float2 b, float) { return b.x; }
__device__ __forceinline__ float2 beta_of(float2 b, float2) { return b; }

// Register tile of a thread.  f32 keeps row pairs packed for fma.rn.f32x2:
// rows 2p and 2p+1 of a column share one 64-bit register pair, the A pair
// comes straight from the 16-byte shared load and the X value is duplicated
// once per k; complex64 keeps plain complex accumulators.
template <typename E, int RM, int RN> struct AccTile;
template <int RM, int RN>
struct AccTile<float, RM, RN> {
    f32x2 v[RM / 2][RN];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < RM / 2; ++i)
#pragma unroll
            for (int j = 0; j < RN; ++j) v[i][j] = 0ull;
    }
    // a: RM values in 16-byte chunks (as loaded), x: RN values
    __device__ __forceinline__ void fma(const float4 (&a)[RM / 4], const float (&x)[RN]) {
#pragma unroll
        for (int j = 0; j < RN; ++j) {
            const f32x2 xd = pack2(x[j], x[j]);
#pragma unroll
            for (int q = 0; q < RM / 4; ++q) {
                const ulonglong2 ap = *reinterpret_cast<const ulonglong2 *>(&a[q]);
                v[2 * q][j] = ffma2(ap.x, xd, v[2 * q][j]);
                v[2 * q + 1][j] = ffma2(ap.y, xd, v[2 * q + 1][j]);
            }
        }
    }
    __device__ __forceinline__ float get(int i, int j) const {
        float lo, hi;
        unpack2(v[i / 2][j], lo, hi);
        return (i & 1) ? hi : lo;
    }
};
template <int RM, int RN>
struct AccTile<float2, RM, RN> {
    float2 v[RM][RN];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
            for (int j = 0; j < RN; ++j) v[i][j] = make_float2(0.f, 0.f);
    }
    __device__ __forceinline__ void fma(const float4 (&a)[RM / 2], const float2 (&x)[RN]) {
#pragma unroll
        for (int i = 0; i < RM; ++i) {
            const float2 ai = reinterpret_cast<const float2 *>(&a[i / 2])[i & 1];
#pragma unroll
            for (int j = 0; j < RN; ++j) v[i][j] = fma_(ai, x[j], v[i][j]);
        }
    }
    __device__ __forceinline__ float2 get(int i, int j) const { return v[i][j]; }
};

template <typename E, bool SMALL>
__global__ void __launch_bounds__(256) sp_update_kernel(const SpArgs g) {
    using Tl = SpTile<E, SMALL>;
    constexpr int VE = Tl::VE, RM = Tl::RM, RN = Tl::RN, BK = Tl::BK, STAGES = Tl::STAGES;
    constexpr int BM = Tl::BM, BN = Tl::BN;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    E *As = reinterpret_cast<E *>(smem_raw);                      // [STAGES][BK][BM]
    E *Xs = As + STAGES * Tl::A_STAGE;                            // [STAGES][BK][BN]

    const E *A = static_cast<const E *>(g.A) + (int64_t)blockIdx.z * g.sA;
    const E *X = static_cast<const E *>(g.X) + (int64_t)blockIdx.z * g.sX;
    E *Cm = static_cast<E *>(g.C) + (int64_t)blockIdx.z * g.sC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp & 1, wn = warp >> 1;
    const int lx = lane & 7, ly = lane >> 3;
    const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
    int64_t kend = g.K;
    if (g.k_by_col && n0 + BN < kend) kend = n0 + BN;
    const int nk = (int)((kend + BK - 1) / BK);

    // one stage: A chunk rows are contiguous (column-major), X chunk columns
    // are contiguous (row-major)
    auto load_stage = [&](int kt, int s) {
        const int64_t k0 = (int64_t)kt * BK;
        E *as = As + s * Tl::A_STAGE;
        E *xs = Xs + s * Tl::X_STAGE;
        constexpr int A_CHUNKS = BK * BM / VE, X_CHUNKS = BK * BN / VE;
#pragma unroll
        for (int c = tid; c < A_CHUNKS; c += 256) {
            const int kk = c / (BM / VE), r = (c % (BM / VE)) * VE;
            const int64_t gr = m0 + r;
            int bytes = 0;
            if (gr < g.M && k0 + kk < kend) bytes = (int)((g.M - gr < VE ? g.M - gr : VE) * sizeof(E));
            const E *src = bytes ? A + (k0 + kk) * g.lda + gr : A;
            cp_async16_zfill(as + kk * BM + r, src, bytes);
        }
#pragma unroll
        for (int c = tid; c < X_CHUNKS; c += 256) {
            const int kk = c / (BN / VE), col = (c % (BN / VE)) * VE;
            const int64_t gc = n0 + col;
            int bytes = 0;
            if (gc < g.N && k0 + kk < kend) bytes = (int)((g.N - gc < VE ? g.N - gc : VE) * sizeof(E));
            const E *src = bytes ? X + (k0 + kk) * g.ldx + gc : X;
            cp_async16_zfill(xs + kk * BN + col, src, bytes);
        }
    };

    AccTile<E, RM, RN> acc;
    acc.zero();

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nk) load_stage(s, s);
        cp_async_commit();
    }

    // fragment offsets inside a stage
    const int a_off = wm * Tl::WM + lx * VE;  // + q * 8 * VE
    const int x_off = wn * Tl::WN + ly * VE;  // + q * 4 * VE

    for (int kt = 0; kt < nk; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {
            const int nxt = kt + STAGES - 1;
            if (nxt < nk) load_stage(nxt, nxt % STAGES);
            cp_async_commit();
        }
        const E *as = As + (kt % STAGES) * Tl::A_STAGE;
        const E *xs = Xs + (kt % STAGES) * Tl::X_STAGE;
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float4 a[RM / VE];
            E x[RN];
#pragma unroll
            for (int q = 0; q < RM / VE; ++q)
                a[q] = *reinterpret_cast<const float4 *>(as + kk * BM + a_off + q * 8 * VE);
#pragma unroll
            for (int q = 0; q < RN / VE; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(xs + kk * BN + x_off + q * 4 * VE);
                const E *e = reinterpret_cast<const E *>(&v);
#pragma unroll
                for (int u = 0; u < VE; ++u) x[q * VE + u] = e[u];
            }
            acc.fma(a, x);
        }
    }
    cp_async_wait_all();

    // epilogue: C = beta*C + gamma*acc, column by column (a thread's rows
    // come in chunks of VE consecutive rows: one 16-byte access where aligned)
    const E beta = beta_of(g.beta, E{});
    const E gamma = beta_of(g.gamma, E{});
    const bool bz = g.beta_zero != 0;
    const bool vec_ok = ((g.ldc * (int64_t)sizeof(E)) % 16 == 0) &&
                        ((reinterpret_cast<uintptr_t>(Cm) & 15) == 0);
#pragma unroll
    for (int j = 0; j < RN; ++j) {
        const int64_t gc = n0 + wn * Tl::WN + (j / VE) * 4 * VE + ly * VE + (j % VE);
        if (gc >= g.N) continue;
        E *ccol = Cm + gc * g.ldc;
#pragma unroll
        for (int q = 0; q < RM / VE; ++q) {
            const int64_t gr0 = m0 + wm * Tl::WM + q * 8 * VE + lx * VE;
            if (vec_ok && gr0 + VE <= g.M) {
                float4 v = bz ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4 *>(ccol + gr0);
                E *e = reinterpret_cast<E *>(&v);
#pragma unroll
                for (int u = 0; u < VE; ++u) {
                    const E t = mul(gamma, acc.get(q * VE + u, j));
                    e[u] = bz ? t : fma_(beta, e[u], t);
                }
                *reinterpret_cast<float4 *>(ccol + gr0) = v;
            } else {
#pragma unroll
                for (int u = 0; u < VE; ++u)
                    if (gr0 + u < g.M) {
                        const E t = mul(gamma, acc.get(q * VE + u, j));
                        ccol[gr0 + u] = bz ? t : fma_(beta, ccol[gr0 + u], t);
                    }
            }
        }
    }
}

}  // namespace trsm
