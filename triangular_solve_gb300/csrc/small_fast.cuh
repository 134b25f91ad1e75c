// Fast small-regime kernel for aligned, full-size systems (m == M, column-
// major, leading dimensions and base pointers 16-byte aligned), the shape of
// every batched small workload.
//
// Versus the general kernel (small_kernels.cuh):
//  * staging moves 16-byte chunks with cp.async: one warp per column of L's
//    packed lower part, flat chunks for the RHS -- no per-element index math;
//  * RHS columns sit in shared memory with a stride of M + 16/sizeof(T)
//    elements (an odd number of 16-byte units), so a thread per column
//    reads its column with conflict-free LDS.128;
//  * a thread solves CPT columns (2 for f32): every broadcast L load feeds
//    CPT times as many FMAs;
//  * X goes from registers straight to global memory with 16-byte stores.
#pragma once

#include <string.h>

#include <type_traits>

#include "internal.h"
#include "small_kernels.cuh"
#include "small_launch.cuh"
#include "mbarrier.cuh"

namespace trsm {

template <typename T, int M, int W>
struct FastImage {
    static constexpr int V = Vec<T>::kN;          // elements per 16 bytes
    static constexpr int kLs = Packed<T, M>::kSize;
    static constexpr int kBld = M + V;            // padded RHS column stride
    static constexpr int kElems = kLs + M + W * kBld;  // multiple of V
    static_assert(kElems % V == 0 && kLs % V == 0 && M % V == 0, "16-byte alignment of the image");
};

// b[c][i] -= col[i] * x[c] for rows i in [FROM, RC), c < CPT.
template <typename T, int RC, int FROM, int CPT>
__device__ __forceinline__ void update_rows_cpt(const T *__restrict__ col, const T (&x)[CPT], T (&b)[CPT][RC]) {
    constexpr int V = Vec<T>::kN;
#pragma unroll
    for (int g0 = 0; g0 < RC; g0 += V) {
        if (g0 + V <= FROM) continue;
        if (g0 >= FROM && g0 + V <= RC) {
            T l[V];
            lds16<T>(col + g0, l);
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int c = 0; c < CPT; ++c) b[c][g0 + v] = fms(l[v], x[c], b[c][g0 + v]);
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (g0 + v >= FROM && g0 + v < RC) {
                    const T l = col[g0 + v];
#pragma unroll
                    for (int c = 0; c < CPT; ++c) b[c][g0 + v] = fms(l, x[c], b[c][g0 + v]);
                }
        }
    }
}

template <typename T, int M, int RC, int CPT, int CH, int KK>
struct FastDiag {
    static __device__ __forceinline__ void run(const T *__restrict__ Ls, const T *__restrict__ dinv,
                                               T (&b)[CPT][RC]) {
        if constexpr (KK < RC) {
            constexpr int k = CH * RC + KK;
            const T d = dinv[k];
            T x[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                x[c] = mul(b[c][KK], d);
                b[c][KK] = x[c];
            }
            update_rows_cpt<T, RC, KK + 1, CPT>(Packed<T, M>::col(Ls, k) + CH * RC, x, b);
            FastDiag<T, M, RC, CPT, CH, KK + 1>::run(Ls, dinv, b);
        }
    }
};

// Chunk CH of RC rows of the thread's CPT columns: earlier chunks' solved
// rows are read back from the staged columns (bs[c]), the chunk is solved,
// written back for later chunks and stored to global memory.
template <typename T, int M, int RC, int CPT, int CH>
struct FastChunks {
    static __device__ __forceinline__ void run(const T *__restrict__ Ls, const T *__restrict__ dinv, T *(&bs)[CPT],
                                               T *(&gout)[CPT], const T alpha, const bool alpha_one) {
        if constexpr (CH < M / RC) {
            constexpr int V = Vec<T>::kN;
            T b[CPT][RC];
            if (alpha_one) {  // uniform: no multiply at all (3% of the FP64 work)
#pragma unroll
                for (int c = 0; c < CPT; ++c)
#pragma unroll
                    for (int g0 = 0; g0 < RC; g0 += V) {
                        T v[V];
                        lds16<T>(bs[c] + CH * RC + g0, v);
#pragma unroll
                        for (int u = 0; u < V; ++u) b[c][g0 + u] = v[u];
                    }
            } else {
#pragma unroll
                for (int c = 0; c < CPT; ++c)
#pragma unroll
                    for (int g0 = 0; g0 < RC; g0 += V) {
                        T v[V];
                        lds16<T>(bs[c] + CH * RC + g0, v);
#pragma unroll
                        for (int u = 0; u < V; ++u) b[c][g0 + u] = mul(alpha, v[u]);
                    }
            }
            // rows solved by earlier chunks: a rolled loop (unrolled by 4),
            // so the code stays small enough for the instruction cache
#pragma unroll 4
            for (int k = 0; k < CH * RC; ++k) {
                T x[CPT];
#pragma unroll
                for (int c = 0; c < CPT; ++c) x[c] = bs[c][k];
                update_rows_cpt<T, RC, 0, CPT>(Packed<T, M>::col(Ls, k) + CH * RC, x, b);
            }
            FastDiag<T, M, RC, CPT, CH, 0>::run(Ls, dinv, b);
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                if (gout[c] == nullptr) continue;
#pragma unroll
                for (int g0 = 0; g0 < RC; g0 += V) {
                    float4 v;
                    T *e = reinterpret_cast<T *>(&v);
#pragma unroll
                    for (int u = 0; u < V; ++u) e[u] = b[c][g0 + u];
                    *reinterpret_cast<float4 *>(gout[c] + CH * RC + g0) = v;
                    if (CH + 1 < M / RC && bs[c] != gout[c]) *reinterpret_cast<float4 *>(bs[c] + CH * RC + g0) = v;
                }
            }
            FastChunks<T, M, RC, CPT, CH + 1>::run(Ls, dinv, bs, gout, alpha, alpha_one);
        }
    }
};

// f32 path on paired FMAs (fma.rn.f32x2).  A thread's column c keeps rows
// 2p and 2p+1 packed in bp[c][p].  Step k: x = b_k / L_kk; the partner row of
// a pair that straddles the diagonal gets one scalar FMA; every later pair
// gets one paired FMA whose L operand (L_2p,k, L_2p+1,k) comes straight from
// a 16- or 8-byte shared load and whose X operand is (-x, -x).
template <int M, int CPT, int KK>
struct FastDiagF2 {
    static __device__ __forceinline__ void run(const float *__restrict__ Ls, const float *__restrict__ dinv,
                                               f32x2 (&bp)[CPT][M / 2]) {
        if constexpr (KK < M) {
            constexpr int pk = KK / 2, half = KK % 2;
            const float d = dinv[KK];
            const float *col = Packed<float, M>::col(Ls, KK);
            f32x2 nx[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float lo, hi, x;
                unpack2(bp[c][pk], lo, hi);
                if constexpr (half == 0) {
                    x = lo * d;
                    lo = x;
                    if constexpr (KK + 1 < M) hi = fmaf(-col[KK + 1], x, hi);
                } else {
                    x = hi * d;
                    hi = x;
                }
                bp[c][pk] = pack2(lo, hi);
                nx[c] = pack2(-x, -x);
            }
#pragma unroll
            for (int p = pk + 1; p < M / 2; ++p) {
                if ((p & 1) && p - 1 >= pk + 1) continue;  // done with its even partner
                if (!(p & 1) && p + 1 < M / 2) {
                    const ulonglong2 l = *reinterpret_cast<const ulonglong2 *>(col + 2 * p);
#pragma unroll
                    for (int c = 0; c < CPT; ++c) {
                        bp[c][p] = ffma2(l.x, nx[c], bp[c][p]);
                        bp[c][p + 1] = ffma2(l.y, nx[c], bp[c][p + 1]);
                    }
                } else {
                    const f32x2 l = *reinterpret_cast<const f32x2 *>(col + 2 * p);
#pragma unroll
                    for (int c = 0; c < CPT; ++c) bp[c][p] = ffma2(l, nx[c], bp[c][p]);
                }
            }
            FastDiagF2<M, CPT, KK + 1>::run(Ls, dinv, bp);
        }
    }
};

template <int M, int CPT>
__device__ __forceinline__ void fast_solve_f32x2(const float *__restrict__ Ls, const float *__restrict__ dinv,
                                                 float *(&bs)[CPT], float *(&gout)[CPT], const float alpha) {
    f32x2 bp[CPT][M / 2];
    const f32x2 a2 = pack2(alpha, alpha);
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int p = 0; p < M / 2; p += 2) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(bs[c] + 2 * p);
            bp[c][p] = ffma2(a2, v.x, 0ull);
            bp[c][p + 1] = ffma2(a2, v.y, 0ull);
        }
    FastDiagF2<M, CPT, 0>::run(Ls, dinv, bp);
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        if (gout[c] == nullptr) continue;
#pragma unroll
        for (int p = 0; p < M / 2; p += 2)
            *reinterpret_cast<ulonglong2 *>(gout[c] + 2 * p) = make_ulonglong2(bp[c][p], bp[c][p + 1]);
    }
}

// ---------------------------------------------------------------------------
// f32 kernel with the right-hand side in registers.  Thread (s, g) owns
// columns g and g + W/2 of system s and loads them with 16-byte global loads
// straight into packed row pairs (no shared staging, so a system needs only
// its packed L and the reciprocal diagonal on chip).  The diagonal advances
// two rows at a time: the 2 x 2 block [[L_kk, 0], [L_k+1,k, L_k+1,k+1]]
// is solved on the pair in registers, then every later pair takes two paired
// FMAs, one per column of the block.
// ---------------------------------------------------------------------------
template <int M>
struct RegImage {
    static constexpr int kLs = Packed<float, M>::kSize;
    static constexpr int kElems = kLs + M;  // + reciprocals; multiple of 4
    static_assert(kElems % 4 == 0, "16-byte aligned images");
};

// Pairs p in [P0, P0 + 2*NG) of one k-pair step, loads first: all 16-byte
// loads of the batch are issued before the first FMA that needs them, so
// the shared-memory latency is paid once per batch rather than per pair.
template <int NG, int CPT>
__device__ __forceinline__ void pair_batch(const float *__restrict__ c0, const float *__restrict__ c1, int p0,
                                           const f32x2 (&n0)[CPT], const f32x2 (&n1)[CPT], f32x2 *bp0,
                                           f32x2 *bp1) {
    ulonglong2 l0[NG], l1[NG];
#pragma unroll
    for (int q = 0; q < NG; ++q) {
        l0[q] = *reinterpret_cast<const ulonglong2 *>(c0 + 2 * (p0 + 2 * q));
        l1[q] = *reinterpret_cast<const ulonglong2 *>(c1 + 2 * (p0 + 2 * q));
    }
#pragma unroll
    for (int q = 0; q < NG; ++q) {
        const int p = p0 + 2 * q;
        bp0[p] = ffma2(l1[q].x, n1[0], ffma2(l0[q].x, n0[0], bp0[p]));
        bp0[p + 1] = ffma2(l1[q].y, n1[0], ffma2(l0[q].y, n0[0], bp0[p + 1]));
        if constexpr (CPT == 2) {
            bp1[p] = ffma2(l1[q].x, n1[1], ffma2(l0[q].x, n0[1], bp1[p]));
            bp1[p + 1] = ffma2(l1[q].y, n1[1], ffma2(l0[q].y, n0[1], bp1[p + 1]));
        }
    }
}

template <int M, int KP, int CPT = 2>
struct RegDiag2 {
    static __device__ __forceinline__ void run(const float *__restrict__ Ls, const float *__restrict__ dinv,
                                               f32x2 (&bp)[CPT][M / 2]) {
        if constexpr (2 * KP < M) {
            constexpr int k0 = 2 * KP, k1 = k0 + 1;
            const float d0 = dinv[k0], d1 = dinv[k1];
            const float *c0 = Packed<float, M>::col(Ls, k0);
            const float *c1 = Packed<float, M>::col(Ls, k1);
            const float l10 = c0[k1];
            f32x2 n0[CPT], n1[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float b0, b1;
                unpack2(bp[c][KP], b0, b1);
                const float x0 = b0 * d0;
                const float x1 = fmaf(-l10, x0, b1) * d1;
                bp[c][KP] = pack2(x0, x1);
                n0[c] = pack2(-x0, -x0);
                n1[c] = pack2(-x1, -x1);
            }
            // a single pair at an odd index first, then 16-byte groups of two
            // pairs, loaded in batches of up to 8 groups
            constexpr int PF = KP + 1;
            constexpr bool odd = (PF & 1) && PF < M / 2;
            if constexpr (odd) {
                const f32x2 l0 = *reinterpret_cast<const f32x2 *>(c0 + 2 * PF);
                const f32x2 l1 = *reinterpret_cast<const f32x2 *>(c1 + 2 * PF);
#pragma unroll
                for (int c = 0; c < CPT; ++c) bp[c][PF] = ffma2(l1, n1[c], ffma2(l0, n0[c], bp[c][PF]));
            }
            constexpr int PG = odd ? PF + 1 : PF;  // first even pair
            constexpr int NGT = (M / 2 - PG) / 2;   // groups of two pairs
            constexpr int BATCH = CPT == 2 ? 4 : 8;
            f32x2 *b1 = CPT == 2 ? bp[CPT - 1] : nullptr;
            if constexpr (NGT > 0) pair_batch<(NGT < BATCH ? NGT : BATCH), CPT>(c0, c1, PG, n0, n1, bp[0], b1);
            if constexpr (NGT > BATCH)
                pair_batch<(NGT - BATCH < BATCH ? NGT - BATCH : BATCH), CPT>(c0, c1, PG + 2 * BATCH, n0, n1, bp[0], b1);
            if constexpr (NGT > 2 * BATCH)
                pair_batch<(NGT - 2 * BATCH < BATCH ? NGT - 2 * BATCH : BATCH), CPT>(c0, c1, PG + 4 * BATCH, n0, n1,
                                                                                   bp[0], b1);
            if constexpr (NGT > 3 * BATCH)
                pair_batch<NGT - 3 * BATCH, CPT>(c0, c1, PG + 6 * BATCH, n0, n1, bp[0], b1);
            RegDiag2<M, KP + 1, CPT>::run(Ls, dinv, bp);
        }
    }
};
static_assert(64 / 2 <= 8 * 4 * 2, "at most four batches of groups per step");

template <int M, int W, int SPC>
__global__ void __launch_bounds__(SPC *(W / 2), 3) small_reg_f32_kernel(const SmallGeom g, const float alpha) {
    using Img = RegImage<M>;
    using P = Packed<float, M>;
    constexpr int G = W / 2;  // threads per system
    constexpr int NT = SPC * G;
    constexpr int NWARPS = (NT + 31) / 32;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *base = reinterpret_cast<float *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j0 = blockIdx.y * W;
    const int64_t sys0 = (int64_t)blockIdx.x * SPC;
    const int nsys = (int)min((int64_t)SPC, g.batch - sys0);
    const float *Ag = static_cast<const float *>(g.A);
    float *Bg = static_cast<float *>(g.B);

    // the thread's two columns, straight into registers (issued first so
    // their latency overlaps the staging of L)
    const int s = tid / G, gi = tid - s * G;
    const bool active = s < nsys;
    f32x2 bp[2][M / 2];
    float *gcol[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int j = j0 + gi + c * G;
        gcol[c] = (active && j < g.n) ? Bg + (sys0 + s) * g.sB + (int64_t)j * g.ldb : nullptr;
#pragma unroll
        for (int p = 0; p < M / 2; p += 2) {
            ulonglong2 v = make_ulonglong2(0ull, 0ull);
            if (gcol[c]) v = *reinterpret_cast<const ulonglong2 *>(gcol[c] + 2 * p);
            bp[c][p] = v.x;
            bp[c][p + 1] = v.y;
        }
    }
    // L's packed lower part: one warp per column, lanes over 16-byte chunks
    for (int cidx = warp; cidx < nsys * M; cidx += NWARPS) {
        const int q = cidx / M, k = cidx - q * M;
        const float *src = Ag + (sys0 + q) * g.sA + (int64_t)k * g.lda + P::s(k);
        float *dst = base + q * Img::kElems + P::off(k);
        const int nch = (M - P::s(k)) / 4;
        for (int e = lane; e < nch; e += 32) cp_async<16>(dst + e * 4, src + e * 4);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int e = tid; e < nsys * M; e += NT) {
        const int q = e / M, k = e - q * M;
        float *img = base + q * Img::kElems;
        img[Img::kLs + k] = 1.0f / img[P::off(k) + (k - P::s(k))];
    }
    __syncthreads();
    if (!active) return;
    const float *Ls = base + s * Img::kElems;
    const f32x2 a2 = pack2(alpha, alpha);
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int p = 0; p < M / 2; ++p) bp[c][p] = ffma2(a2, bp[c][p], 0ull);
    RegDiag2<M, 0>::run(Ls, Ls + Img::kLs, bp);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (gcol[c] == nullptr) continue;
#pragma unroll
        for (int p = 0; p < M / 2; p += 2)
            *reinterpret_cast<ulonglong2 *>(gcol[c] + 2 * p) = make_ulonglong2(bp[c][p], bp[c][p + 1]);
    }
}

// ---------------------------------------------------------------------------
// Persistent f32 kernel: pairs of warps stream their own sequence of work
// items (system, 64-column slice) through a two-stage shared-memory ring.
// The two warps of a pair share the staged L and take 32 columns each (one
// per lane).  While a pair solves item i from one stage (columns in
// registers, as above), the cp.async copies of item i+1 fill the other stage,
// so HBM traffic and the substitution overlap inside every pair; pairs
// synchronise with their own named barrier, never the whole CTA.  The CTA
// first builds a table of the 16-byte chunks of L's packed lower part
// (column, first row, shared offset), which turns the L copy into a flat
// loop.
// ---------------------------------------------------------------------------
template <int M>
struct PipeStage {
    static constexpr int kLs = Packed<float, M>::kSize;
    static constexpr int kBld = M + 4;                 // padded column stride
    static constexpr int kElems = kLs + M + 64 * kBld;  // L, reciprocals, 64 columns
    static constexpr int kChunks = kLs / 4;            // 16-byte chunks of L
    static_assert(kElems % 4 == 0, "16-byte aligned stages");
};

struct ChunkEntry {
    unsigned short k, row0, dst;  // column, first row, offset in the packed image
};

constexpr int kPipePairs = 4;

__device__ __forceinline__ void pair_barrier(int pair) {
    asm volatile("bar.sync %0, 64;\n" ::"r"(pair + 1) : "memory");
}

template <int M>
__global__ void __launch_bounds__(64 * kPipePairs, 1) small_pipe_f32_kernel(const SmallGeom g, const float alpha,
                                                                          const int64_t items) {
    using St = PipeStage<M>;
    using P = Packed<float, M>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *stages = reinterpret_cast<float *>(smem_raw);  // [pairs][2][kElems]
    ChunkEntry *tab = reinterpret_cast<ChunkEntry *>(stages + kPipePairs * 2 * St::kElems);
    const int tid = threadIdx.x;
    const int pair = tid >> 6, pt = tid & 63;  // thread within the pair = its column

    // chunk table: column k owns (M - s(k)) / 4 chunks starting at row s(k)
    for (int k = tid; k < M; k += blockDim.x) {
        const int nch = (M - P::s(k)) / 4;
        const int first = P::off(k) / 4;  // chunks before column k
        for (int q = 0; q < nch; ++q) {
            ChunkEntry e;
            e.k = (unsigned short)k;
            e.row0 = (unsigned short)(P::s(k) + 4 * q);
            e.dst = (unsigned short)(P::off(k) + 4 * q);
            tab[first + q] = e;
        }
    }
    __syncthreads();

    const int slices = (g.n + 63) / 64;
    const int64_t gp = (int64_t)blockIdx.x * kPipePairs + pair;
    const int64_t np = (int64_t)gridDim.x * kPipePairs;
    const float *Ag = static_cast<const float *>(g.A);
    float *Bg = static_cast<float *>(g.B);
    float *my = stages + pair * 2 * St::kElems;

    auto issue = [&](int64_t item, float *st) {
        const int64_t sys = item / slices;
        const int j0 = (int)(item - sys * slices) * 64;
        const float *A = Ag + sys * g.sA;
        for (int e = pt; e < St::kChunks; e += 64) {
            const ChunkEntry c = tab[e];
            cp_async<16>(st + c.dst, A + (int64_t)c.k * g.lda + c.row0);
        }
        const float *B = Bg + sys * g.sB;
        float *bs = st + St::kLs + M;
        constexpr int CPC = M / 4;  // chunks per column
        for (int e = pt; e < 64 * CPC; e += 64) {
            const int j = e / CPC, q = e - j * CPC;
            float *dst = bs + j * St::kBld + 4 * q;
            if (j0 + j < g.n) cp_async<16>(dst, B + (int64_t)(j0 + j) * g.ldb + 4 * q);
            else *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };

    int64_t item = gp;
    if (item < items) issue(item, my);
    cp_async_commit();
    for (int it = 0; item < items; ++it, item += np) {
        float *cur = my + (it & 1) * St::kElems;
        const int64_t next = item + np;
        if (next < items) issue(next, my + ((it + 1) & 1) * St::kElems);
        cp_async_commit();
        cp_async_wait<1>();
        pair_barrier(pair);
        if (pt < M) cur[St::kLs + pt] = 1.0f / cur[P::off(pt) + (pt - P::s(pt))];
        pair_barrier(pair);

        const int64_t sys = item / slices;
        const int j = (int)(item - sys * slices) * 64 + pt;
        const float *bcol = cur + St::kLs + M + pt * St::kBld;
        f32x2 bp[1][M / 2];
        const f32x2 a2 = pack2(alpha, alpha);
#pragma unroll
        for (int p = 0; p < M / 2; p += 2) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(bcol + 2 * p);
            bp[0][p] = ffma2(a2, v.x, 0ull);
            bp[0][p + 1] = ffma2(a2, v.y, 0ull);
        }
        RegDiag2<M, 0, 1>::run(cur, cur + St::kLs, bp);
        if (j < g.n) {
            float *gcol = Bg + sys * g.sB + (int64_t)j * g.ldb;
#pragma unroll
            for (int p = 0; p < M / 2; p += 2)
                *reinterpret_cast<ulonglong2 *>(gcol + 2 * p) = make_ulonglong2(bp[0][p], bp[0][p + 1]);
        }
        pair_barrier(pair);  // the stage is refilled by the prefetch two items ahead
    }
    cp_async_wait_all();
}

// ---------------------------------------------------------------------------
// Persistent f32 kernel on the TMA engine (m = 32, 48, 64).  Same work split
// as the kernel above -- pairs of warps, a two-stage ring per pair, one
// column per lane in registers -- but every HBM transfer is a tiled tensor
// copy, off the load/store pipe that the L broadcasts keep busy:
//   in   the lower 32 x 32 boxes of L (3 for m = 64) and the RHS slice as
//        32-row x 64-column boxes, with the 128-byte shared-memory swizzle
//        (16-byte chunk q of a 128-byte line c sits at chunk q ^ (c % 8)), so
//        that a lane reading its own column meets no bank conflicts;
//   out  X is written back over its RHS column and leaves as the same boxes
//        (the tensor store clips columns past n and rows past m).
// Per item that is a handful of copies, where per-column copies would be
// limited by the copy engine's rate for small transfers.  Shapes the tensor
// maps cannot describe take the kernel above.
// ---------------------------------------------------------------------------
template <int M>
struct SwzStage {
    static_assert(M == 32 || M == 48 || M == 64, "32-row boxes");
    static constexpr int NR = (M + 31) / 32;                   // 32-row blocks
    static constexpr int kLFloats = NR * (NR + 1) / 2 * 1024;  // lower boxes of L, 4 KB each
    static constexpr int kBFloats = NR * 2048;                 // RHS boxes, 8 KB each
    static constexpr int kElems = kLFloats + kBFloats;
    static constexpr uint32_t kBytes = 4u * kElems;
    // rows 4q .. 4q+3 of column k of L (box of row block q/8 and column block k/32)
    static __host__ __device__ constexpr int loff(int k, int q) {
        return ((q / 8) * (q / 8 + 1) / 2 + k / 32) * 1024 + (k % 32) * 32 + (((q % 8) ^ (k % 8)) * 4);
    }
    static __host__ __device__ constexpr int lel(int i, int k) { return loff(k, i / 4) + i % 4; }
    // rows 4q .. 4q+3 of column c of the RHS slice
    static __device__ __forceinline__ int boff(int c, int q) {
        return kLFloats + (q / 8) * 2048 + c * 32 + (((q % 8) ^ (c & 7)) * 4);
    }
};

// The substitution of RegDiag2 (two rows per step, CPT columns per lane) on
// the swizzled image; 1/L_kk comes from lane k % 32 of dlo (k < 32) or dhi.
template <int M, int KP, int CPT>
struct SwzDiag2 {
    static __device__ __forceinline__ void run(const float *__restrict__ st, float dlo, float dhi,
                                               f32x2 (&bp)[CPT][M / 2]) {
        using S = SwzStage<M>;
        if constexpr (2 * KP < M) {
            constexpr int k0 = 2 * KP, k1 = k0 + 1;
            const float d0 = __shfl_sync(0xffffffffu, k0 < 32 ? dlo : dhi, k0 % 32);
            const float d1 = __shfl_sync(0xffffffffu, k1 < 32 ? dlo : dhi, k1 % 32);
            const float l10 = st[S::lel(k1, k0)];
            f32x2 n0[CPT], n1[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float b0, b1;
                unpack2(bp[c][KP], b0, b1);
                const float x0 = b0 * d0;
                const float x1 = fmaf(-l10, x0, b1) * d1;
                bp[c][KP] = pack2(x0, x1);
                n0[c] = pack2(-x0, -x0);
                n1[c] = pack2(-x1, -x1);
            }
            constexpr int PF = KP + 1;
            constexpr bool odd = (PF & 1) && PF < M / 2;
            if constexpr (odd) {  // rows 2PF, 2PF+1: the upper half of chunk PF/2
                const f32x2 l0 = *reinterpret_cast<const f32x2 *>(st + S::loff(k0, PF / 2) + 2);
                const f32x2 l1 = *reinterpret_cast<const f32x2 *>(st + S::loff(k1, PF / 2) + 2);
#pragma unroll
                for (int c = 0; c < CPT; ++c) bp[c][PF] = ffma2(l1, n1[c], ffma2(l0, n0[c], bp[c][PF]));
            }
            constexpr int Q0 = (odd ? PF + 1 : PF) / 2, NQ = M / 4 - Q0;  // whole chunks left
            constexpr int QB = CPT == 2 ? 4 : 8;                          // chunks per load batch
#pragma unroll
            for (int qb = 0; qb < NQ; qb += QB) {
                ulonglong2 a[QB], b[QB];
#pragma unroll
                for (int u = 0; u < QB; ++u)
                    if (qb + u < NQ) {
                        a[u] = *reinterpret_cast<const ulonglong2 *>(st + S::loff(k0, Q0 + qb + u));
                        b[u] = *reinterpret_cast<const ulonglong2 *>(st + S::loff(k1, Q0 + qb + u));
                    }
#pragma unroll
                for (int u = 0; u < QB; ++u)
                    if (qb + u < NQ) {
                        const int p = 2 * (Q0 + qb + u);
#pragma unroll
                        for (int c = 0; c < CPT; ++c) {
                            bp[c][p] = ffma2(b[u].x, n1[c], ffma2(a[u].x, n0[c], bp[c][p]));
                            bp[c][p + 1] = ffma2(b[u].y, n1[c], ffma2(a[u].y, n0[c], bp[c][p + 1]));
                        }
                    }
            }
            SwzDiag2<M, KP + 1, CPT>::run(st, dlo, dhi, bp);
        }
    }
};

// WPI warps per item: 2 (a pair, one column per lane: 8 warps per SM) or 1
// (two columns per lane, half the L broadcasts per item, 4 warps per SM);
// units of WPI warps per CTA, as many as the stages fit.  Measured on GB300:
// pairs are faster at m = 64, single warps at m = 32 and 48.
template <int WPI>
struct TmaUnits {
    static constexpr int kUnits = WPI == 2 ? kPipePairs : 4;
    static constexpr int kThreads = 32 * WPI * kUnits;
};

__device__ __forceinline__ void unit_sync(int unit, int nthreads) {
    if (nthreads == 32) __syncwarp();
    else asm volatile("bar.sync %0, %1;\n" ::"r"(unit + 1), "r"(nthreads) : "memory");
}

__device__ __forceinline__ bool unit_any(int unit, int nthreads, bool flag) {
    if (nthreads == 32) return __any_sync(0xffffffffu, flag);
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)flag), "r"(unit + 1), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int M, int WPI>
__global__ void __launch_bounds__(TmaUnits<WPI>::kThreads, 1)
    small_tma_f32_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                         const int n, const float alpha, const int64_t items, int *status,
                         const uint32_t wait_limit) {
    using S = SwzStage<M>;
    constexpr int NR = S::NR, UNITS = TmaUnits<WPI>::kUnits, UT = 32 * WPI, CPT = 2 / WPI;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[UNITS][2];
    const int tid = threadIdx.x;
    const int unit = tid / UT, wu = (tid / 32) % WPI, lane = tid & 31;
    const bool leader = (tid % UT) == 0;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // the swizzle pattern repeats every 1024 bytes
    float *my = reinterpret_cast<float *>(smem_raw + (sbase - raw)) + unit * 2 * S::kElems;
    if (tid < 2 * UNITS) mbar_init(smem_u32(&full_bar[tid >> 1][tid & 1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    __syncthreads();

    const int slices = (n + 63) / 64;
    auto issue = [&](int64_t item, int s) {  // the unit's leader
        const int sys = (int)(item / slices);
        const int j0 = (int)(item - (int64_t)sys * slices) * 64;
        const uint32_t bar = smem_u32(&full_bar[unit][s]);
        const uint32_t st = smem_u32(my + s * S::kElems);
        mbar_expect_tx(bar, S::kBytes);
        for (int rb = 0; rb < NR; ++rb)
            for (int cb = 0; cb <= rb; ++cb)
                tma_load_3d(st + 4u * (uint32_t)((rb * (rb + 1) / 2 + cb) * 1024), &mapA, 32 * rb, 32 * cb, sys, bar);
        for (int rb = 0; rb < NR; ++rb)
            tma_load_3d(st + 4u * (uint32_t)(S::kLFloats + rb * 2048), &mapB, 32 * rb, j0, sys, bar);
    };

    int64_t item = (int64_t)blockIdx.x * UNITS + unit;
    const int64_t step = (int64_t)gridDim.x * UNITS;
    if (leader && item < items) issue(item, 0);
    for (int it = 0; item < items; ++it, item += step) {
        const int s = it & 1;
        const bool more = item + step < items;
        if (leader && more) {
            bulk_wait_read<0>();  // the last item's stores have read stage s^1
            issue(item + step, s ^ 1);
        }
        // wait_limit polls (kWaitLimit unless lowered through
        // trsm_set_wait_limit); the waits that drain the copies in flight
        // below keep the full limit
        const bool ok = mbar_wait_n(smem_u32(&full_bar[unit][s]), (uint32_t)(it >> 1) & 1u, wait_limit);
        if (unit_any(unit, UT, !ok)) {
            // a copy never completed: report, let the copies in flight land, stop
            if (leader) record_timeout(status);
            mbar_wait(smem_u32(&full_bar[unit][s]), (uint32_t)(it >> 1) & 1u);
            if (more) mbar_wait(smem_u32(&full_bar[unit][s ^ 1]), (uint32_t)((it + 1) >> 1) & 1u);
            break;
        }
        float *cur = my + s * S::kElems;
        const float dlo = 1.0f / cur[S::lel(lane, lane)];
        const float dhi = (M > 32 && lane + 32 < M) ? 1.0f / cur[S::lel(lane + 32, lane + 32)] : 0.f;
        int col[CPT];  // columns of the slice
#pragma unroll
        for (int c = 0; c < CPT; ++c) col[c] = 32 * (wu + c) + lane;
        f32x2 bp[CPT][M / 2];
        const f32x2 a2 = pack2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int q = 0; q < M / 4; ++q) {
                const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(cur + S::boff(col[c], q));
                bp[c][2 * q] = ffma2(a2, v.x, 0ull);
                bp[c][2 * q + 1] = ffma2(a2, v.y, 0ull);
            }
        SwzDiag2<M, 0, CPT>::run(cur, dlo, dhi, bp);
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
            for (int q = 0; q < M / 4; ++q)
                *reinterpret_cast<ulonglong2 *>(cur + S::boff(col[c], q)) =
                    make_ulonglong2(bp[c][2 * q], bp[c][2 * q + 1]);
        fence_proxy_async_smem();
        unit_sync(unit, UT);
        if (leader) {
            const int sys = (int)(item / slices);
            const int j0 = (int)(item - (int64_t)sys * slices) * 64;
            for (int rb = 0; rb < NR; ++rb)
                tma_store_3d(&mapB, 32 * rb, j0, sys, smem_u32(cur + S::kLFloats + rb * 2048));
            bulk_commit();
        }
    }
    if (leader) bulk_wait<0>();  // every store complete before the CTA's shared memory goes away
}

// CTA: SPC systems x (W / CPT) threads each.  Thread g of a system owns
// columns g + c*(W/CPT), c < CPT, of the CTA's column slice.
// Shared image of a system whose RHS stays in global memory: packed L and the
// reciprocal diagonal, rounded up to 16 bytes.
template <typename T, int M>
constexpr int fast_direct_image() {
    constexpr int V = Vec<T>::kN;
    return (Packed<T, M>::kSize + M + V - 1) / V * V;
}

template <typename T, int M, int W, int CPT, int RC, int SPC>
__global__ void __launch_bounds__(SPC *(W / CPT)) small_fast_kernel(const SmallGeom g, const T alpha) {
    using Img = FastImage<T, M, W>;
    using P = Packed<T, M>;
    constexpr int V = Img::V;
    // FP64 types read their RHS straight from global memory, chunk by chunk
    // (the FP64 rate hides the latency), so a system needs only L on chip
    // and several systems share an SM
    constexpr bool kDirect = std::is_same<T, double>::value || std::is_same<T, double2>::value;
    constexpr int kImg = kDirect ? fast_direct_image<T, M>() : Img::kElems;
    constexpr int G = W / CPT;           // threads per system
    constexpr int NT = SPC * G;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *base = reinterpret_cast<T *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NWARPS = (NT + 31) / 32;
    const int j0 = blockIdx.y * W;
    const int64_t sys0 = (int64_t)blockIdx.x * SPC;
    const int nsys = (int)min((int64_t)SPC, g.batch - sys0);
    const T *Ag = static_cast<const T *>(g.A);
    T *Bg = static_cast<T *>(g.B);

    // L: one warp per column, lanes over the column's 16-byte chunks
    for (int cidx = warp; cidx < nsys * M; cidx += NWARPS) {
        const int s = cidx / M, k = cidx - s * M;
        const T *src = Ag + (sys0 + s) * g.sA + (int64_t)k * g.lda + P::s(k);
        T *dst = base + s * kImg + P::off(k);
        const int nch = (M - P::s(k)) / V;
        for (int q = lane; q < nch; q += 32) cp_async<16>(dst + q * V, src + q * V);
    }
    // RHS slice: flat 16-byte chunks; columns past n are zero-filled
    constexpr int CH_PER_COL = M / V;
    for (int e = tid; !kDirect && e < nsys * W * CH_PER_COL; e += NT) {
        const int s = e / (W * CH_PER_COL), r = e - s * (W * CH_PER_COL);
        const int j = r / CH_PER_COL, q = r - j * CH_PER_COL;
        T *dst = base + s * Img::kElems + Img::kLs + M + j * Img::kBld + q * V;
        if (j0 + j < g.n) cp_async<16>(dst, Bg + (sys0 + s) * g.sB + (int64_t)(j0 + j) * g.ldb + q * V);
        else *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    cp_async_wait_all();
    __syncthreads();
    // reciprocals of the diagonal (row k of packed column k)
    for (int e = tid; e < nsys * M; e += NT) {
        const int s = e / M, k = e - s * M;
        T *img = base + s * kImg;
        img[Img::kLs + k] = recip(img[P::off(k) + (k - P::s(k))]);
    }
    __syncthreads();

    const int s = tid / G, gi = tid - s * G;
    if (s >= nsys) return;
    const T *Ls = base + s * kImg;
    const T *dinv = Ls + Img::kLs;
    T *bs[CPT];
    T *gout[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int j = gi + c * G;
        gout[c] = (j0 + j < g.n) ? Bg + (sys0 + s) * g.sB + (int64_t)(j0 + j) * g.ldb : nullptr;
        bs[c] = kDirect ? gout[c] : base + s * Img::kElems + Img::kLs + M + j * Img::kBld;
    }
    if (kDirect && gout[0] == nullptr) return;  // one column per thread: past n
    if constexpr (std::is_same<T, float>::value && CPT == 2 && RC == M)
        fast_solve_f32x2<M, CPT>(Ls, dinv, bs, gout, alpha);
    else
        FastChunks<T, M, RC, CPT, 0>::run(Ls, dinv, bs, gout, alpha, is_one(alpha));
}

}  // namespace trsm

namespace trsm {

constexpr int kFastNotApplicable = -100000;

template <typename T, int M, int W, int CPT, int RC>
static int launch_fast_mw(const SmallGeom &g, T alpha, cudaStream_t st) {
    constexpr int G = W / CPT;
    constexpr bool kDirect = std::is_same<T, double>::value || std::is_same<T, double2>::value;
    constexpr size_t per =
        (size_t)(kDirect ? fast_direct_image<T, M>() : FastImage<T, M, W>::kElems) * sizeof(T);
    constexpr int SPC_T = 128 / G > 0 ? 128 / G : 1;               // ~128 threads per CTA
    constexpr int SPC_S = (int)((220 * 1024) / per) > 0 ? (int)((220 * 1024) / per) : 1;
    // FP64 types: one system per CTA, so that the scheduler balances the
    // last wave system by system (several CTAs share an SM)
    constexpr int SPC = kDirect ? 1 : (SPC_T < SPC_S ? SPC_T : SPC_S);
    constexpr size_t smem = (size_t)SPC * per;
    static_assert(smem <= 227 * 1024, "fast small kernel shared memory");
    auto kern = small_fast_kernel<T, M, W, CPT, RC, SPC>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_status(e);
    }
    const dim3 grid((unsigned)((g.batch + SPC - 1) / SPC), (unsigned)((g.n + W - 1) / W));
    kern<<<grid, SPC * G, smem, st>>>(g, alpha);
    return launch_status();
}

template <int M, int W>
static int launch_reg_f32(const SmallGeom &g, float alpha, cudaStream_t st) {
    constexpr int G = W / 2;
    constexpr int SPC = 128 / G;
    constexpr size_t smem = (size_t)SPC * RegImage<M>::kElems * sizeof(float);
    auto kern = small_reg_f32_kernel<M, W, SPC>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_status(e);
    }
    const dim3 grid((unsigned)((g.batch + SPC - 1) / SPC), (unsigned)((g.n + W - 1) / W));
    kern<<<grid, SPC * G, smem, st>>>(g, alpha);
    return launch_status();
}

template <int M>
static int launch_pipe_f32(const SmallGeom &g, float alpha, cudaStream_t st) {
    using St = PipeStage<M>;
    constexpr size_t smem = (size_t)kPipePairs * 2 * St::kElems * sizeof(float) + St::kChunks * sizeof(ChunkEntry);
    static_assert(smem <= 227 * 1024, "pipelined kernel shared memory");
    auto kern = small_pipe_f32_kernel<M>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_status(e);
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t items = g.batch * ((g.n + 63) / 64);
    const int64_t per_cta = kPipePairs;
    int64_t ctas = (items + per_cta - 1) / per_cta;
    if (ctas > sms) ctas = sms;  // persistent: one CTA per SM
    kern<<<(unsigned)ctas, 64 * kPipePairs, smem, st>>>(g, alpha, items);
    return launch_status();
}

// The TMA kernel when the tensor maps accept the strides (base, leading
// dimensions and batch strides 16-byte multiples, batch < 2^31);
// kFastNotApplicable otherwise.
constexpr int kTmaNotApplicable = -100001;

template <int M, int WPI>
static int launch_tma_f32(const SmallGeom &g, float alpha, cudaStream_t st) {
    using S = SwzStage<M>;
    if (g.batch >= (int64_t(1) << 31)) return kTmaNotApplicable;
    CUtensorMap ma, mb;
    const uint64_t da[3] = {(uint64_t)M, (uint64_t)M, (uint64_t)g.batch};
    const uint64_t sa[2] = {(uint64_t)g.lda * 4, (uint64_t)g.sA * 4};
    const uint32_t ba[3] = {32, 32, 1};
    if (encode_f32_map(&ma, g.A, 3, da, sa, ba, true)) return kTmaNotApplicable;
    const uint64_t db[3] = {(uint64_t)M, (uint64_t)g.n, (uint64_t)g.batch};
    const uint64_t sb[2] = {(uint64_t)g.ldb * 4, (uint64_t)g.sB * 4};
    const uint32_t bb[3] = {32, 64, 1};
    if (encode_f32_map(&mb, g.B, 3, db, sb, bb, true)) return kTmaNotApplicable;
    constexpr int UNITS = TmaUnits<WPI>::kUnits;
    constexpr size_t smem = (size_t)UNITS * 2 * S::kElems * sizeof(float) + 1024;
    static_assert(smem <= 227 * 1024, "TMA kernel shared memory");
    auto kern = small_tma_f32_kernel<M, WPI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_status(e);
    int *status = nullptr;
    const int rc = device_status_word(&status);
    if (rc) return rc;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 152;
    const int64_t items = g.batch * ((g.n + 63) / 64);
    int64_t ctas = (items + UNITS - 1) / UNITS;
    if (ctas > sms) ctas = sms;  // persistent: one CTA per SM
    kern<<<(unsigned)ctas, TmaUnits<WPI>::kThreads, smem, st>>>(ma, mb, g.n, alpha, items, status,
                                                                 first_wait_limit());
    return launch_status();
}

template <typename T, int M>
static int launch_fast_m(const SmallGeom &g, T alpha, cudaStream_t st) {
    if constexpr (std::is_same<T, float>::value) {
        if (g.n <= 16) return launch_reg_f32<M, 32>(g, alpha, st);
        if constexpr (M >= 16) {
            // many items: a persistent kernel; a handful: one CTA per few
            // systems finishes sooner
            if (g.batch * ((g.n + 63) / 64) >= 4 * 152) {
                if constexpr (M % 16 == 0 && M >= 32) {
                    const int rc = launch_tma_f32<M, (M == 64 ? 2 : 1)>(g, alpha, st);
                    if (rc != kTmaNotApplicable) return rc;
                }
                return launch_pipe_f32<M>(g, alpha, st);
            }
        }
        if (g.n <= 32) return launch_reg_f32<M, 32>(g, alpha, st);
        return launch_reg_f32<M, 64>(g, alpha, st);
    }
    if constexpr (std::is_same<T, double>::value || std::is_same<T, double2>::value) {
        // too few systems to occupy every SM: spread their columns instead
        // (a whole system on one SM is bound by that SM's FP64 rate)
        static int sms = 0;
        if (sms == 0) {
            int dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (sms <= 0) sms = 152;
        }
        if (g.batch * ((g.n + 63) / 64) < 2 * sms) return launch_rowlane_split_m<T, M>(g, alpha, sms, st);
    }
    constexpr int CPT = std::is_same<T, float>::value ? 2 : 1;
    // row chunk: 16 rows for the complex types, 32 for f64; only the chunk's
    // own triangle is unrolled (a whole unrolled 64-row triangle of c64
    // outgrows the instruction cache: "no instruction" stalls dominated)
    constexpr int RCX = Elem<T>::kComplex ? 16 : 32;
    constexpr int RC = (M > RCX && M % RCX == 0) ? RCX : M;
    if (g.n <= 32) return launch_fast_mw<T, M, 32, CPT, RC>(g, alpha, st);
    return launch_fast_mw<T, M, 64, CPT, RC>(g, alpha, st);
}

// m = 128 (batches of medium systems, which otherwise run one by one through
// the blocked path): the chunked kernel alone -- 32-row chunks for the real
// types, 16 for the complex ones, one CTA holding up to three f32 systems or
// one system of the other types (L packed in shared memory: 66-132 KB).
template <typename T>
static int launch_fast_128(const SmallGeom &g, T alpha, cudaStream_t st) {
    constexpr int CPT = std::is_same<T, float>::value ? 2 : 1;
    constexpr int RC = Elem<T>::kComplex ? 16 : 32;
    if (g.n <= 32) return launch_fast_mw<T, 128, 32, CPT, RC>(g, alpha, st);
    return launch_fast_mw<T, 128, 64, CPT, RC>(g, alpha, st);
}

// The fast kernel's preconditions: column-major, m one of the compiled
// sizes, every column and system start 16-byte aligned.  Returns
// kFastNotApplicable otherwise (the general kernel then runs).
template <typename T>
int launch_fast_typed(const SmallArgs &a, cudaStream_t st) {
    const int64_t s = (int64_t)sizeof(T);
    const bool al = a.layout == 0 && ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) == 0 &&
                    (a.lda * s) % 16 == 0 && (a.ldb * s) % 16 == 0 && (a.strideA * s) % 16 == 0 &&
                    (a.strideB * s) % 16 == 0 && a.n > 8;
    if (!al) return kFastNotApplicable;
    SmallGeom g;
    g.m = (int)a.m; g.n = (int)a.n; g.layout = 0;
    g.A = a.A; g.lda = a.lda; g.sA = a.strideA;
    g.B = a.B; g.ldb = a.ldb; g.sB = a.strideB;
    g.batch = a.batch; g.spc = 0; g.w = 0;
    T alpha;
    memcpy(&alpha, a.alpha, sizeof(T));
    switch (a.m) {
        case 8: return launch_fast_m<T, 8>(g, alpha, st);
        case 16: return launch_fast_m<T, 16>(g, alpha, st);
        case 32: return launch_fast_m<T, 32>(g, alpha, st);
        case 48: return launch_fast_m<T, 48>(g, alpha, st);
        case 64: return launch_fast_m<T, 64>(g, alpha, st);
        case 128: return launch_fast_128<T>(g, alpha, st);
        default: return kFastNotApplicable;
    }
}

}  // namespace trsm
