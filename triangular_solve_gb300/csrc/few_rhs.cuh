// Few right-hand sides (n <= 8) on one large system.
//
// With a handful of columns the blocked path's GEMMs have no width: every
// product is a thin matrix-vector product bound by reading L once from HBM,
// and the per-block-row launches dominate.  This path keeps the blocked
// algorithm of "Hierarchical Shared Memory-Aware Optimization for TRSM on GPU
// Platforms" -- the diagonal blocks inverted up front (W_t = D_t^{-1}), then
// per block row t
//     x_t = W_t (alpha b_t - sum_{s<t} L_ts x_s)
// -- but runs all block rows in one cooperatively launched persistent
// kernel.  The CTA that owns block row t streams its tiles L_ts (s < t) and
// then W_t on chip, independently of the solve, folds tile s in as soon as
// the owner of block row s has published x_s, and publishes x_t in turn.
// The reduction sum_{s<t} L_ts x_s is spread over the owners of the block
// rows below, in parallel; only one 128 x 128 product and the application of
// W_t per block row lie on the dependency chain.
//
// Roles inside a CTA (warp specialised, no CTA-wide barrier after set-up):
//   warp 0    issues the TMA tensor copies of the tiles, 128 rows x KC
//             columns at a time, into a ring of mbarrier-tracked stages;
//   warp 1    polls each block row's published x_s and stages it in a small
//             ring of slots, a few tiles ahead of the consumers;
//   warps 2-9 consume: two threads a row, each accumulating its row of
//             L_ts x_s over half of each chunk's columns; the halves meet
//             once per product in shared memory.  In f32 with n = 1 the
//             tile on the chain, L_{t,t-1}, and W_t are moved to registers
//             before x_{t-1} arrives.
// In the cluster form (CL) consecutive block rows sit in a cluster and x_t
// also goes straight into the next CTA's shared memory (see the kernel).
// Every wait is bounded; on expiry the CTA records TRSM_ERR_DEVICE_TIMEOUT,
// lets its copies and hand-offs in flight land and returns.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "mbarrier.cuh"

namespace trsm {

// right-hand sides it takes: kFewMaxN (internal.h, with the workspace size)

// Block rows: 128.  (256 halves the chain of block rows, but then the tile
// and W_t a step needs -- 512 KB in f32 -- no longer fit on chip ahead of
// x_s, and streaming them lengthens every step: measured slower.)
template <typename T>
constexpr int few_nb() {
    return (int)kFewNb;
}

// CL: the cluster form (x_{t-1} handed over in shared memory, see the
// kernel), which needs one more slot.
template <typename T, bool CL>
struct FewCfg {
    static constexpr int NB = few_nb<T>();
    static constexpr int HALVES = 256 / NB;                         // consumer threads per row
    static constexpr int Q = (int)sizeof(T) / 4;                    // floats per element
    static constexpr int BR = 256 / Q < NB ? 256 / Q : NB;          // rows per tensor-copy box
    static constexpr int KC = 32768 / (NB * (int)sizeof(T));        // columns per 32 KB chunk
    static constexpr int KPT = NB / KC;                             // chunks per tile
    static constexpr int kChunk = NB * KC;                          // elements per chunk
    static constexpr int XS = sizeof(T) >= 16 ? 2 : 4;              // x slots
    static constexpr int kSlot = NB * kFewMaxN;                     // elements per x slot (and rbuf, part, dsx)
    static constexpr size_t kFixed = (size_t)(XS + 2 + (CL ? 1 : 0)) * kSlot * sizeof(T);
    static constexpr int ST = (int)((220 * 1024 - kFixed) / (kChunk * sizeof(T)));  // ring stages
    static constexpr size_t kSmem = (size_t)ST * kChunk * sizeof(T) + kFixed + 1024;
    static_assert(KC * NB * (int)sizeof(T) == 32768 && KPT >= 2 && KC % (2 * HALVES) == 0, "32 KB chunks");
    static_assert(HALVES == 2, "two threads a row");
    static_assert(ST >= 3, "ring depth");
};

__device__ __forceinline__ float add2_(float a, float b) { return a + b; }
__device__ __forceinline__ double add2_(double a, double b) { return a + b; }
__device__ __forceinline__ float2 add2_(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ double2 add2_(double2 a, double2 b) { return make_double2(a.x + b.x, a.y + b.y); }

// Publication of x_t without a separate flag: the published copy starts as
// all-ones words (memset before the launch), a pattern no arithmetic result
// takes (NaNs are stored in canonical form), and every word is written once,
// by a single store, so a reader that sees no all-ones word has the values.
// That saves the flag's round trip on the chain of block rows.
__device__ __forceinline__ bool unset_word(float v) { return __float_as_uint(v) == 0xffffffffu; }
__device__ __forceinline__ bool unset_word(double v) { return __double_as_longlong(v) == -1ll; }
__device__ __forceinline__ bool is_unset(float v) { return unset_word(v); }
__device__ __forceinline__ bool is_unset(double v) { return unset_word(v); }
__device__ __forceinline__ bool is_unset(float2 v) { return unset_word(v.x) || unset_word(v.y); }
__device__ __forceinline__ bool is_unset(double2 v) { return unset_word(v.x) || unset_word(v.y); }
__device__ __forceinline__ float canon(float v) { return v != v ? __uint_as_float(0x7fffffffu) : v; }
__device__ __forceinline__ double canon(double v) { return v != v ? __longlong_as_double(0x7fffffffffffffffll) : v; }
__device__ __forceinline__ float2 canon(float2 v) { return make_float2(canon(v.x), canon(v.y)); }
__device__ __forceinline__ double2 canon(double2 v) { return make_double2(canon(v.x), canon(v.y)); }
// The published copy is written and polled with relaxed gpu-scope accesses:
// a plain load in a polling loop may legally be hoisted out of it (another
// thread's store is then a data race), a relaxed one may not, and it reads
// the L2's current value.  Each component is one single-copy-atomic access.
__device__ __forceinline__ float load_fresh(const float *p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];\n" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ double load_fresh(const double *p) {
    double v;
    asm volatile("ld.relaxed.gpu.global.f64 %0, [%1];\n" : "=d"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float2 load_fresh(const float2 *p) {
    float2 v;
    asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ double2 load_fresh(const double2 *p) {
    double2 v;
    asm volatile("ld.relaxed.gpu.global.v2.f64 {%0, %1}, [%2];\n" : "=d"(v.x), "=d"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void store_published(float *p, float v) {
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;\n" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void store_published(double *p, double v) {
    asm volatile("st.relaxed.gpu.global.f64 [%0], %1;\n" ::"l"(p), "d"(v) : "memory");
}
__device__ __forceinline__ void store_published(float2 *p, float2 v) {
    asm volatile("st.relaxed.gpu.global.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ void store_published(double2 *p, double2 v) {
    asm volatile("st.relaxed.gpu.global.v2.f64 [%0], {%1, %2};\n" ::"l"(p), "d"(v.x), "d"(v.y) : "memory");
}
// Every thread of every CTA of the cluster (a CTA of its own without one).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;\n" ::: "memory");
}
// v into the same shared-memory location of CTA `rank` of the cluster,
// completing that CTA's mbarrier at bar's address by sizeof(v) bytes.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_async_remote(float *p, float v, uint64_t *bar, uint32_t rank) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];\n" ::"r"(
                     cluster_addr(p, rank)),
                 "r"(__float_as_uint(v)), "r"(cluster_addr(bar, rank))
                 : "memory");
}
__device__ __forceinline__ void st_async_remote(double *p, double v, uint64_t *bar, uint32_t rank) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];\n" ::"r"(
                     cluster_addr(p, rank)),
                 "l"(__double_as_longlong(v)), "r"(cluster_addr(bar, rank))
                 : "memory");
}
__device__ __forceinline__ void st_async_remote(float2 *p, float2 v, uint64_t *bar, uint32_t rank) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];\n" ::"r"(
                     cluster_addr(p, rank)),
                 "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(cluster_addr(bar, rank))
                 : "memory");
}
__device__ __forceinline__ void st_async_remote(double2 *p, double2 v, uint64_t *bar, uint32_t rank) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b64 [%0], {%1, %2}, [%3];\n" ::"r"(
                     cluster_addr(p, rank)),
                 "l"(__double_as_longlong(v.x)), "l"(__double_as_longlong(v.y)), "r"(cluster_addr(bar, rank))
                 : "memory");
}

// two consecutive elements of shared memory (8-byte aligned pairs of f32,
// 16-byte of the others) in one access where the width allows
__device__ __forceinline__ void load_pair(const float *p, float &a, float &b) {
    const float2 v = *reinterpret_cast<const float2 *>(p);
    a = v.x, b = v.y;
}
__device__ __forceinline__ void load_pair(const double *p, double &a, double &b) {
    const double2 v = *reinterpret_cast<const double2 *>(p);
    a = v.x, b = v.y;
}
__device__ __forceinline__ void load_pair(const float2 *p, float2 &a, float2 &b) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    a = make_float2(v.x, v.y), b = make_float2(v.z, v.w);
}
__device__ __forceinline__ void load_pair(const double2 *p, double2 &a, double2 &b) { a = p[0], b = p[1]; }
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }

// NC: right-hand sides the registers and loops are sized for (n <= NC; the
// launcher picks the smallest of 1, 2, 4, 8): a guarded loop over a fixed
// eight would still issue the idle columns' FMAs, which on the FP64 pipe
// cost as much as the real ones.
template <typename T, int NC, bool CL>
__global__ void __launch_bounds__(320, 1)
    few_rhs_kernel(const __grid_constant__ CUtensorMap mapL, const __grid_constant__ CUtensorMap mapW, int64_t m,
                   int n, T *B, int64_t ldb, const T alpha, T *xpub, int *status, const int64_t poll_limit) {
    using C = FewCfg<T, CL>;
    constexpr int NB = C::NB, KC = C::KC, KPT = C::KPT, ST = C::ST, XS = C::XS, BR = C::BR, Q = C::Q;
    // f32 with one right-hand side holds the tile on the chain and W_t in
    // registers (see the consumers); W_t then comes first in a block row's
    // stream
    constexpr bool kReg = std::is_same<T, float>::value && NC == 1;
    constexpr int KH = KC / C::HALVES;  // columns of a chunk per thread
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full[ST], empty[ST], xfull[XS], xempty[XS], dsbar;
    __shared__ volatile int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    T *ring = reinterpret_cast<T *>(smem_raw + (((raw + 1023u) & ~1023u) - raw));  // [ST][chunk]
    T *xs = ring + ST * C::kChunk;                                                  // [XS][8][NB]
    T *rbuf = xs + XS * C::kSlot;                                                   // [8][NB]: r_t
    T *part = rbuf + C::kSlot;                                                      // [8][NB]
    T *dsx = part + C::kSlot;  // [8][NB]: x_{t-1}, written by the CTA before this one in the cluster
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t tb = (m + NB - 1) / NB;
    // In a cluster of K CTAs (consecutive block rows, the grid a multiple of
    // K), every CTA but the cluster's first receives x_{t-1} straight into
    // its shared memory from the CTA that solves it (st.async, completing
    // dsbar), and every CTA but the last sends x_t on: the hop through L2
    // remains only at cluster boundaries and for the block rows further down.
    // (kept in shared memory, read where needed: the f32 consumers' registers
    // are full with L_{t,t-1} and W_t)
    __shared__ int sh_rank, sh_left, sh_right;
    if constexpr (CL)
        for (int e = tid; e < C::kSlot; e += blockDim.x) dsx[e] = zero_of<T>();  // columns >= n stay zero
    if (tid == 0) {
        if constexpr (CL) {
            uint32_t crank, csize;
            asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(crank));
            asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(csize));
            sh_rank = (int)crank;
            sh_left = crank > 0;
            sh_right = crank + 1 < csize;
            mbar_init(smem_u32(&dsbar), 1);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 8);
        }
        for (int s = 0; s < XS; ++s) {
            mbar_init(smem_u32(&xfull[s]), 1);
            mbar_init(smem_u32(&xempty[s]), 8);
        }
        abort_flag = 0;
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    __syncthreads();
    // every CTA of the cluster has its barriers ready before any st.async
    if constexpr (CL) cluster_sync_all();

    auto copies = [&]() {
        // ---------------------------------------------------------- copies
        if (lane != 0) return;
        int64_t g = 0;  // chunks issued
        bool ok = true;
        for (int64_t t = blockIdx.x; t < tb && ok; t += gridDim.x) {
            const int64_t nch = (t + 1) * KPT;  // tiles s < t of L and W_t (first when kReg, else last)
            for (int64_t c = 0; c < nch; ++c, ++g) {
                const int stage = (int)(g % ST);
                if ((g >= ST && !mbar_wait(smem_u32(&empty[stage]), (uint32_t)((g / ST - 1) & 1))) ||
                    abort_flag) {
                    ok = false;
                    break;
                }
                const uint32_t bar = smem_u32(&full[stage]);
                mbar_expect_tx(bar, (uint32_t)(C::kChunk * sizeof(T)));
                const int64_t s = kReg ? (c < KPT ? t : c / KPT - 1) : c / KPT;
                const int k0 = (int)(c % KPT) * KC;
                const uint32_t dst = smem_u32(ring + stage * C::kChunk);
                for (int b = 0; b < NB / BR; ++b) {
                    // box b: rows b*BR.. of the chunk, KC columns, at b*BR*KC elements
                    const uint32_t d = dst + (uint32_t)(b * BR * KC * (int)sizeof(T));
                    if (s < t)
                        tma_load_3d(d, &mapL, (int)((t * NB + b * BR) * Q), (int)(s * NB + k0), 0, bar);
                    else
                        tma_load_3d(d, &mapW, b * BR * Q, (int)(t * NB + k0), 0, bar);
                }
            }
        }
        if (!ok) {
            // the copies issued last may still be landing: wait for them
            record_timeout(status);
            abort_flag = 1;
            for (int64_t h = (g > ST ? g - ST : 0); h < g; ++h)
                mbar_wait(smem_u32(&full[h % ST]), (uint32_t)((h / ST) & 1));
        }
    };

    auto poller = [&]() {
        // ---------------------------------------------------------- x_s
        constexpr int kPollE = NB * NC / 32;                        // elements a lane polls
        constexpr bool kPollTwo = kPollE * sizeof(T) <= 64;         // two polls held in registers
        constexpr long long kPollGap = 600;                         // cycles, about half an L2 round trip
        int64_t gx = 0;
        for (int64_t t = blockIdx.x; t < tb; t += gridDim.x) {
            for (int64_t s = 0; s < t; ++s) {
                if (CL && s == t - 1 && sh_left) continue;  // x_{t-1} arrives in dsx
                const int slot = (int)(gx % XS);
                bool ok = true;
                if (gx >= XS) ok = mbar_wait(smem_u32(&xempty[slot]), (uint32_t)((gx / XS - 1) & 1));
                // poll the published x_s (column cc at xpub[(s n + cc) NB ..])
                // until no word is unset; lane element q: e = lane + 32 q
                T *dst = xs + slot * C::kSlot;
                const T *src = xpub + s * (int64_t)n * NB;
                auto issue = [&](T (&v)[kPollE]) {
#pragma unroll
                    for (int q = 0; q < kPollE; ++q) {
                        const int e = lane + 32 * q, cc = e / NB;
                        v[q] = cc < n ? load_fresh(src + cc * NB + e % NB) : zero_of<T>();
                    }
                };
                auto landed = [&](const T (&v)[kPollE]) {
                    bool mine = true;
#pragma unroll
                    for (int q = 0; q < kPollE; ++q) mine = mine && !is_unset(v[q]);
                    if (!__all_sync(0xffffffffu, mine)) return false;
#pragma unroll
                    for (int q = 0; q < kPollE; ++q) {
                        const int e = lane + 32 * q;
                        dst[(e / NB) * NB + e % NB] = v[q];
                    }
                    return true;
                };
                int64_t polls = 0;
                if constexpr (kPollTwo) {
                    // two polls in flight, issued about half a round trip
                    // apart (the first pair split by a short spin, then each
                    // poll reissued as soon as its check comes back)
                    T va[kPollE], vb[kPollE];
                    if (ok) {
                        issue(va);
                        const long long t0 = clock64();
                        while (clock64() - t0 < kPollGap) {
                        }
                    }
                    while (ok) {
                        issue(vb);
                        if (landed(va)) break;
                        issue(va);
                        if (landed(vb)) break;
                        if ((polls += 2) > poll_limit || abort_flag) ok = false;
                    }
                } else {
                    // too wide to hold in registers: staged as it is read
                    while (ok) {
                        bool mine = true;
                        for (int e = lane; e < NB * NC; e += 32) {
                            const int cc = e / NB, i = e % NB;
                            T v = zero_of<T>();
                            if (cc < n) {
                                v = load_fresh(src + cc * NB + i);
                                if (is_unset(v)) mine = false;
                            }
                            dst[cc * NB + i] = v;
                        }
                        if (__all_sync(0xffffffffu, mine)) break;
                        if (++polls > poll_limit || abort_flag) ok = false;
                    }
                }
                if (!ok || abort_flag) {
                    if (lane == 0) {
                        record_timeout(status);
                        abort_flag = 1;
                    }
                    return;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&xfull[slot]));
                ++gx;
            }
        }
    };

    auto consume = [&]() {
    // -------------------------------------------------------------- consume
    // Every consumer warp runs the same sequence of stage releases and
    // consumer barriers whatever happens: after a failed wait (abort_flag set)
    // the warps stop waiting and computing and only walk the sequence, so the
    // barriers still match; the copy warp stops issuing once it sees abort_flag
    // and waits for the copies it has in flight before it returns.
    // Two threads per row, each over half of a chunk's columns: a warp
    // covers 32 rows (conflict-free shared-memory reads of the tiles), the
    // halves in warps cw and cw + 4, meeting in shared memory.
    const int ct = tid - 64, row = ct % NB, half = ct / NB;
    const bool wl = lane == 0;
    int64_t g = 0, gx = 0;
    auto fail = [&]() {
        if (!abort_flag) {
            record_timeout(status);
            abort_flag = 1;
        }
    };
    // the halves' sums of a row, in half 0
    auto combine = [&](T (&acc)[NC]) {
        if (half == 1) {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) part[cc * NB + row] = acc[cc];
        }
        consumer_sync();
        if (half == 0) {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) acc[cc] = add2_(acc[cc], part[cc * NB + row]);
        }
    };
    // one chunk of the ring into acc: columns k0.. of the x source ([cc][NB])
    auto chunk = [&](const T *__restrict__ xsrc, int k0, T (&acc)[NC]) {
        const int stage = (int)(g % ST);
        if (!abort_flag && !mbar_wait(smem_u32(&full[stage]), (uint32_t)((g / ST) & 1))) fail();
        if (!abort_flag) {
            const T *ch = ring + stage * C::kChunk;
            T acc2[NC];
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) acc2[cc] = zero_of<T>();
            // element (r, j) of a chunk: box r / BR, column j, row r % BR
            const T *base = ch + (row / BR) * BR * KC + row % BR;
#pragma unroll(NC >= 4 ? 2 : 4)
            for (int jj = 0; jj < KH; jj += 2) {
                const int j = half * KH + jj;
                const T a0 = base[j * BR], a1 = base[(j + 1) * BR];
                const T *xk = xsrc + k0 + j;
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    T x0, x1;
                    load_pair(xk + cc * NB, x0, x1);
                    acc[cc] = fma_(a0, x0, acc[cc]);
                    acc2[cc] = fma_(a1, x1, acc2[cc]);
                }
            }
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) acc[cc] = add2_(acc[cc], acc2[cc]);
        }
        __syncwarp();
        if (wl) mbar_arrive(smem_u32(&empty[stage]));
        ++g;
    };
    // kReg (f32, n = 1): the tile on the chain (L_{t,t-1}) and W_t go to
    // registers while x_{t-1} is still on its way (128 of the 168 registers
    // a thread has with ten warps on an SM), so the chain step reads only x
    // from shared memory.  Chunk kc holds columns kc KC ..: with KC = NB / 2
    // this thread's half is exactly chunk `half`.
    constexpr int HC = kReg ? NB / 2 : 1;
    static_assert(!kReg || (KC == HC && KPT == 2 && BR == NB), "f32 chunks are column halves");
    auto preload = [&](T (&R)[HC]) {
        for (int kc = 0; kc < KPT; ++kc) {
            const int64_t h = g + kc;
            if (!abort_flag && !mbar_wait(smem_u32(&full[h % ST]), (uint32_t)((h / ST) & 1))) fail();
        }
        if (!abort_flag) {
            const T *ch = ring + (int)((g + half) % ST) * C::kChunk + row;
#pragma unroll
            for (int j = 0; j < HC; ++j) R[j] = ch[j * BR];
        } else {
#pragma unroll
            for (int j = 0; j < HC; ++j) R[j] = zero_of<T>();
        }
        __syncwarp();
        if (wl)
            for (int kc = 0; kc < KPT; ++kc) mbar_arrive(smem_u32(&empty[(g + kc) % ST]));
        g += KPT;
    };
    // acc += R . src over this thread's half of the columns (src [cc][NB]);
    // a few partial sums per column keep the FMA chains short
    auto reg_matvec = [&](const T (&R)[HC], const T *__restrict__ src, T (&acc)[NC]) {
        if constexpr (kReg) {
            constexpr int P = NC >= 4 ? 1 : 4 / NC;
            float p[P][NC];
#pragma unroll
            for (int q = 0; q < P; ++q)
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) p[q][cc] = 0.f;
            const float *xb = src + half * HC;
#pragma unroll
            for (int j = 0; j < HC; j += 4) {
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    const float4 v = *reinterpret_cast<const float4 *>(xb + cc * NB + j);
                    p[(j / 4 + 0) % P][cc] = fmaf(R[j], v.x, p[(j / 4 + 0) % P][cc]);
                    p[(j / 4 + 1) % P][cc] = fmaf(R[j + 1], v.y, p[(j / 4 + 1) % P][cc]);
                    p[(j / 4 + 2) % P][cc] = fmaf(R[j + 2], v.z, p[(j / 4 + 2) % P][cc]);
                    p[(j / 4 + 3) % P][cc] = fmaf(R[j + 3], v.w, p[(j / 4 + 3) % P][cc]);
                }
            }
#pragma unroll
            for (int q = 0; q < P; ++q)
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) acc[cc] += p[q][cc];
        }
    };
    T Lreg[HC], Wreg[HC];
    // dsbar: one phase per block row (t >= 1 whenever there is a left neighbour), armed by
    // thread ct 0 at the block row's start -- not after a failure, when the
    // earlier phase may still be open (the end of the kernel drains them)
    uint32_t pass = 0, armed = 0;
    for (int64_t t = blockIdx.x; t < tb; t += gridDim.x, ++pass) {
        const int64_t r0 = t * NB;
        if (CL && ct == 0 && sh_left && !abort_flag) {
            mbar_expect_tx(smem_u32(&dsbar), (uint32_t)(n * NB * (int)sizeof(T)));
            ++armed;
        }
        // alpha b_t, loaded now: off the chain of block rows
        T ab[NC];
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
            ab[cc] = (half == 0 && cc < n && r0 + row < m) ? mul(alpha, B[cc * ldb + r0 + row]) : zero_of<T>();
        T acc[NC];
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) acc[cc] = zero_of<T>();
        const int64_t s_reg = kReg ? t - 1 : t;  // the tile from registers
        if (kReg) preload(Wreg);
        for (int64_t s = 0; s < t; ++s) {
            const bool local = CL && s == t - 1 && sh_left;  // x_s in dsx, not in a slot
            const int slot = (int)(gx % XS);
            if (s == s_reg) preload(Lreg);
            if (local) {
                if (!abort_flag && !mbar_wait(smem_u32(&dsbar), pass & 1u)) fail();
            } else if (!abort_flag && !mbar_wait(smem_u32(&xfull[slot]), (uint32_t)((gx / XS) & 1))) {
                fail();
            }
            const T *xsrc = local ? dsx : xs + slot * C::kSlot;
            if (s == s_reg) {
                if (!abort_flag) reg_matvec(Lreg, xsrc, acc);
            } else {
                for (int kc = 0; kc < KPT; ++kc) chunk(xsrc, kc * KC, acc);
            }
            if (!local) {
                __syncwarp();
                if (wl) mbar_arrive(smem_u32(&xempty[slot]));
                ++gx;
            }
        }
        // every tile is in: r_t = alpha b_t - sum_s L_ts x_s
        combine(acc);
        if (half == 0) {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc)
                rbuf[cc * NB + row] = sub_(ab[cc], acc[cc]);
        }
        consumer_sync();
        // x_t = W_t r_t
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) acc[cc] = zero_of<T>();
        if (kReg) {
            if (!abort_flag) reg_matvec(Wreg, rbuf, acc);
        } else {
            for (int kc = 0; kc < KPT; ++kc) chunk(rbuf, kc * KC, acc);
        }
        combine(acc);
        // X over b_t, and the published copy for the block rows below (also
        // after a failure -- the status word then says the result is void --
        // so that the CTAs waiting on it finish instead of timing out)
        // (and to the next CTA of the cluster, which solves block row t + 1)
        const bool send = CL && t + 1 < tb && sh_right;
        if (half == 0 && r0 + row < m) {
#pragma unroll
            for (int cc = 0; cc < NC; ++cc)
                if (cc < n) {
                    B[cc * ldb + r0 + row] = acc[cc];
                    store_published(xpub + (t * n + cc) * NB + row, canon(acc[cc]));
                    if (send) st_async_remote(dsx + cc * NB + row, acc[cc], &dsbar, (uint32_t)sh_rank + 1);
                }
        }
        consumer_sync();  // rbuf and part are rewritten for the next block row
    }
    // after a failure every hand-off the left neighbour sends (it sends one
    // per block row whatever happens) must still land before this CTA may
    // exit: wait for the open phase, then arm and wait for the rest in order
    if (CL && ct == 0 && sh_left && armed < pass) {
        if (armed > 0) mbar_wait(smem_u32(&dsbar), (armed - 1) & 1u);
        for (uint32_t q = armed; q < pass; ++q) {
            mbar_expect_tx(smem_u32(&dsbar), (uint32_t)(n * NB * (int)sizeof(T)));
            mbar_wait(smem_u32(&dsbar), q & 1u);
        }
    }
    };

    if (warp == 0)
        copies();
    else if (warp == 1)
        poller();
    else
        consume();
    // no CTA leaves while a neighbour may still write into its shared memory
    if constexpr (CL) cluster_sync_all();
}

template <typename T, bool CL>
constexpr size_t few_rhs_smem() {
    return FewCfg<T, CL>::kSmem;
}

}  // namespace trsm
