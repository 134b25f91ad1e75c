// Small-regime TRSM kernels (m <= 64): the whole lower triangle of one
// system and its right-hand-side slice are staged on chip, then solved by
// forward substitution without touching global memory again.
//
// "Hierarchical Shared Memory-Aware Optimization for TRSM on GPU Platforms",
// small-scale regime (m, n <= 64): A is held entirely in shared memory and the
// right-hand side is staged on chip, with the solve overlapped with memory
// traffic.  The pages size this for a 48-64 KB budget (half of B at a time,
// and a seven-stage two-group pipeline for complex double).  On sm_103a a CTA
// may use up to 227 KB, so every type -- complex double included -- stages
// the full lower triangle and the full RHS slice at once, and the overlap
// comes from several CTAs per SM instead of an intra-CTA pipeline.
//
// Two thread mappings:
//  * colreg  (n > 8):  one thread per RHS column.  The thread keeps its
//    column in registers (in row chunks of RC for wide types) and walks the
//    columns of L left to right (x_k = b_k / L_kk, then b_i -= L_ik x_k for
//    i > k).  Every thread of a system reads the same L_ik, so the shared
//    loads are broadcasts and there is no per-row reduction or barrier (the
//    llama.cpp SOLVE_TRI kernel of PR 17457 instead reduces a dot product
//    across a warp and synchronises after every row).
//  * rowlane (n <= 8): one warp per system, lane l owns rows l and l+32 of
//    every column; x_k travels from its owner lane by a register shuffle.
#pragma once

#include "common.cuh"

namespace trsm {

struct SmallGeom {
    int m, n, layout;  // layout: 0 column-major, 1 row-major
    const void *A;
    int64_t lda, sA;
    void *B;
    int64_t ldb, sB;
    int64_t batch;
    int spc;  // systems per CTA
    int w;    // RHS columns per CTA slice (colreg) / register columns (rowlane)
};

// Systems of order m <= 8: one thread per (system, right-hand-side
// column), the column in registers, the triangle read through L1 (a warp's
// threads share a few systems, so most reads are broadcasts), forward
// substitution with the diagonal's reciprocals -- computed once per system
// into shared memory when three or more columns share it (in FP64 the
// reciprocals were most of the work).  Either layout.  At this size a warp
// per system or a CTA per few systems leaves most lanes idle; here every
// thread does a whole column, and the grid is batch x n threads.
constexpr int kTinyM = 8;
template <typename T>
__global__ void __launch_bounds__(256) small_tiny_kernel(const SmallGeom g, const T alpha) {
    constexpr int M = kTinyM, kMaxSys = 256 / 3 + 2;  // systems a CTA touches when n >= 3
    __shared__ T rinv[kMaxSys * M];
    const int64_t total = g.batch * g.n, gid0 = (int64_t)blockIdx.x * 256, gid = gid0 + threadIdx.x;
    const int m = g.m;
    const T *A0 = static_cast<const T *>(g.A);
    // element (i, k): column-major i + k ld, row-major i ld + k
    const int64_t ar = g.layout ? g.lda : 1, ac = g.layout ? 1 : g.lda;
    const int64_t br = g.layout ? g.ldb : 1, bc = g.layout ? 1 : g.ldb;
    const bool shared_rinv = g.n >= 3;
    const int64_t b0 = gid0 / g.n;
    if (shared_rinv) {
        const int64_t last = (gid0 + 255 < total ? gid0 + 255 : total - 1);
        const int nsys = (int)(last / g.n - b0 + 1);
        for (int e = threadIdx.x; e < nsys * M; e += 256) {
            const int k = e % M;
            rinv[e] = k < m ? recip(ldg(A0 + (b0 + e / M) * g.sA + k * (ar + ac))) : zero_of<T>();
        }
        __syncthreads();
    }
    if (gid >= total) return;
    const int64_t b = gid / g.n;
    const int j = (int)(gid - b * g.n);
    const T *A = A0 + b * g.sA;
    T *B = static_cast<T *>(g.B) + b * g.sB;
    T x[M];
#pragma unroll
    for (int i = 0; i < M; ++i) x[i] = i < m ? mul(alpha, B[i * br + j * bc]) : zero_of<T>();
#pragma unroll
    for (int k = 0; k < M; ++k) {
        if (k < m) {
            const T d = shared_rinv ? rinv[(b - b0) * M + k] : recip(ldg(A + k * (ar + ac)));
            x[k] = mul(x[k], d);
#pragma unroll
            for (int i = k + 1; i < M; ++i)
                if (i < m) x[i] = fms(ldg(A + i * ar + k * ac), x[k], x[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < M; ++i)
        if (i < m) B[i * br + j * bc] = x[i];
}

// Vector width (elements per 16-byte shared load).
template <typename T> struct Vec { static constexpr int kN = sizeof(T) >= 16 ? 1 : 16 / (int)sizeof(T); };

// Packed lower triangle in shared memory.  Column k keeps rows
// [s(k), M) with s(k) = k rounded down to the vector width V, so every
// column starts 16-byte aligned and the strictly lower rows k+1.. are read
// with 16-byte broadcast loads.  Rows s(k)..k of column k are never read.
// Column k starts at off(k) = sum_{q<k} (M - s(q)); total (M^2 + M V)/2.
template <typename T, int M>
struct Packed {
    static constexpr int V = Vec<T>::kN;
    static __host__ __device__ constexpr int s(int k) { return (k / V) * V; }
    static __host__ __device__ constexpr int off(int k) {
        // sum_{q<k} s(q) = V * (V a (a-1)/2 + a b),  k = a V + b
        return k * M - V * (V * (k / V) * (k / V - 1) / 2 + (k / V) * (k % V));
    }
    static constexpr int kSize = (M * M + M * V) / 2;
    static_assert(off(M) == kSize, "packed size");
    // pointer p such that p[i] is row i of column k (valid for i >= s(k))
    static __device__ __forceinline__ const T *col(const T *Ls, int k) { return Ls + off(k) - s(k); }
};

// Shared-memory image of one system:
//   Ls   packed strictly-lower columns of L (see Packed); padding rows
//        >= m hold zero; the never-read rows s(k)..k of column k hold zero
//        or, when whole 16-byte groups are copied, the matrix's own values.
//   dinv M reciprocals of the diagonal (zero for padding rows >= m).
//   Bs   w columns of the RHS, column stride M + 1 (odd, so a thread per
//        column reads its own column without bank conflicts).
template <typename T, int M>
struct SmallImage {
    static constexpr int kLs = Packed<T, M>::kSize;
    static constexpr int kBld = M + 1;
    static __host__ __device__ __forceinline__ int elems(int w) {
        const int e = kLs + M + w * kBld;
        constexpr int a = sizeof(T) >= 16 ? 1 : 16 / (int)sizeof(T);
        return (e + a - 1) / a * a;  // keep every system's Ls 16-byte aligned
    }
};

// Cooperative copy of system `sys` into its shared image.  Elements copied
// from memory go through cp.async; the complement is zero-filled with plain
// stores (disjoint addresses, so no ordering is needed between the two).
template <typename T, int M>
__device__ __forceinline__ void stage_system(const SmallGeom &g, T *Ls, T *dinv, T *Bs, int64_t sys,
                                             int j0, int wcols, int tid, int nthr) {
    const T *A = static_cast<const T *>(g.A) + sys * g.sA;
    const T *B = static_cast<const T *>(g.B) + sys * g.sB;
    const int m = g.m;
    const T z = zero_of<T>();
    using P = Packed<T, M>;
    if (g.layout == 0) {
        constexpr int V = P::V, G = M / V;  // elements per 16 bytes, 16-byte groups per full column
        if (V > 1 && m == M && (reinterpret_cast<uintptr_t>(A) & 15) == 0 && g.lda % V == 0) {
            // full-size, aligned: whole 16-byte groups of column k from row
            // s(k) (its rows s(k)..k come along and are never read), a
            // fraction of the element-wise loop's instructions
            for (int e = tid; e < M * G; e += nthr) {
                const int k = e / G, q = e - k * G;
                if (q * V < P::s(k)) continue;
                cp_async<16>(Ls + P::off(k) + (q * V - P::s(k)), A + (int64_t)k * g.lda + q * V);
            }
        } else {
            for (int e = tid; e < M * M; e += nthr) {
                const int k = e / M, i = e - k * M;
                if (i < P::s(k)) continue;
                T *d = Ls + P::off(k) + (i - P::s(k));
                if (i > k && i < m) cp_async<sizeof(T)>(d, A + (int64_t)k * g.lda + i);
                else *d = z;
            }
        }
        for (int e = tid; e < wcols * M; e += nthr) {
            const int c = e / M, i = e - c * M;
            T *d = Bs + c * (M + 1) + i;
            if (i < m) cp_async<sizeof(T)>(d, B + (int64_t)(j0 + c) * g.ldb + i);
            else *d = z;
        }
    } else {
        for (int e = tid; e < M * M; e += nthr) {
            const int i = e / M, k = e - i * M;
            if (i < P::s(k)) continue;
            T *d = Ls + P::off(k) + (i - P::s(k));
            if (i > k && i < m) cp_async<sizeof(T)>(d, A + (int64_t)i * g.lda + k);
            else *d = z;
        }
        for (int e = tid; e < wcols * M; e += nthr) {
            const int i = e / wcols, c = e - i * wcols;
            T *d = Bs + c * (M + 1) + i;
            if (i < m) cp_async<sizeof(T)>(d, B + (int64_t)i * g.ldb + (j0 + c));
            else *d = z;
        }
    }
    for (int e = tid; e < M; e += nthr) dinv[e] = e < m ? recip(ldg(A + (int64_t)e * g.lda + e)) : z;
}

template <typename T, int M>
__device__ __forceinline__ void unstage_system(const SmallGeom &g, const T *Bs, int64_t sys, int j0,
                                               int wcols, int tid, int nthr) {
    T *B = static_cast<T *>(g.B) + sys * g.sB;
    const int m = g.m;
    if (g.layout == 0) {
        for (int e = tid; e < wcols * M; e += nthr) {
            const int c = e / M, i = e - c * M;
            if (i < m) B[(int64_t)(j0 + c) * g.ldb + i] = Bs[c * (M + 1) + i];
        }
    } else {
        for (int e = tid; e < wcols * M; e += nthr) {
            const int i = e / wcols, c = e - i * wcols;
            if (i < m) B[(int64_t)i * g.ldb + (j0 + c)] = Bs[c * (M + 1) + i];
        }
    }
}

template <typename T>
__device__ __forceinline__ void lds16(const T *p, T (&out)[Vec<T>::kN]) {
    if constexpr (Vec<T>::kN == 1) {
        out[0] = *p;
    } else {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        const T *s = reinterpret_cast<const T *>(&v);
#pragma unroll
        for (int q = 0; q < Vec<T>::kN; ++q) out[q] = s[q];
    }
}

// b[ii] -= col[ii] * xk for ii in [FROM, RC).  col is 16-byte aligned; rows
// are read in 16-byte broadcast loads where a whole group is in range.
template <typename T, int RC, int FROM>
__device__ __forceinline__ void update_rows(const T *__restrict__ col, const T xk, T (&b)[RC]) {
    constexpr int V = Vec<T>::kN;
#pragma unroll
    for (int g0 = 0; g0 < RC; g0 += V) {
        if (g0 + V <= FROM) continue;
        if (g0 >= FROM && g0 + V <= RC) {
            T l[V];
            lds16<T>(col + g0, l);
#pragma unroll
            for (int v = 0; v < V; ++v) b[g0 + v] = fms(l[v], xk, b[g0 + v]);
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v)
                if (g0 + v >= FROM && g0 + v < RC) b[g0 + v] = fms(col[g0 + v], xk, b[g0 + v]);
        }
    }
}

// Diagonal-block step kk of a chunk, recursing at compile time so that the
// row range of every update is a constant.
template <typename T, int M, int RC, int CH, int KK>
struct DiagSteps {
    static __device__ __forceinline__ void run(const T *__restrict__ Ls, const T *__restrict__ dinv, T (&b)[RC]) {
        if constexpr (KK < RC) {
            constexpr int k = CH * RC + KK;
            const T xk = mul(b[KK], dinv[k]);
            b[KK] = xk;
            update_rows<T, RC, KK + 1>(Packed<T, M>::col(Ls, k) + CH * RC, xk, b);
            DiagSteps<T, M, RC, CH, KK + 1>::run(Ls, dinv, b);
        }
    }
};

// Solve one column (staged at bs, stride 1) in chunks of RC rows; solved
// chunks are written back to bs, from where later chunks read them.
template <typename T, int M, int RC, int CH>
struct ColumnChunks {
    static __device__ __forceinline__ void run(const T *__restrict__ Ls, const T *__restrict__ dinv, T *bs,
                                               const T alpha) {
        if constexpr (CH < M / RC) {
            T b[RC];
#pragma unroll
            for (int ii = 0; ii < RC; ++ii) b[ii] = mul(alpha, bs[CH * RC + ii]);
#pragma unroll
            for (int k = 0; k < CH * RC; ++k) {
                const T xk = bs[k];
                update_rows<T, RC, 0>(Packed<T, M>::col(Ls, k) + CH * RC, xk, b);
            }
            DiagSteps<T, M, RC, CH, 0>::run(Ls, dinv, b);
#pragma unroll
            for (int ii = 0; ii < RC; ++ii) bs[CH * RC + ii] = b[ii];
            ColumnChunks<T, M, RC, CH + 1>::run(Ls, dinv, bs, alpha);
        }
    }
};

template <typename T, int M, int RC>
__global__ void __launch_bounds__(256) small_colreg_kernel(const SmallGeom g, const T alpha) {
    static_assert(M % RC == 0, "row chunks must tile the column");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *base = reinterpret_cast<T *>(smem_raw);
    const int w = g.w;
    const int per = SmallImage<T, M>::elems(w);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int j0 = blockIdx.y * w;
    const int wcols = min(w, g.n - j0);
    const int64_t sys0 = (int64_t)blockIdx.x * g.spc;
    const int nsys = (int)min((int64_t)g.spc, g.batch - sys0);

    for (int s = 0; s < nsys; ++s) {
        T *Ls = base + s * per;
        stage_system<T, M>(g, Ls, Ls + SmallImage<T, M>::kLs, Ls + SmallImage<T, M>::kLs + M, sys0 + s, j0,
                           wcols, tid, nthr);
    }
    cp_async_wait_all();
    __syncthreads();

    const int s = tid / w, c = tid - s * w;
    if (s < nsys && c < wcols) {
        const T *Ls = base + s * per;
        T *bs = base + s * per + SmallImage<T, M>::kLs + M + c * (M + 1);
        ColumnChunks<T, M, RC, 0>::run(Ls, Ls + SmallImage<T, M>::kLs, bs, alpha);
    }
    __syncthreads();

    for (int q = 0; q < nsys; ++q)
        unstage_system<T, M>(g, base + q * per + SmallImage<T, M>::kLs + M, sys0 + q, j0, wcols, tid, nthr);
}

// ---------------------------------------------------------------- rowlane
__device__ __forceinline__ float shfl(float v, int src) { return __shfl_sync(0xffffffffu, v, src); }
__device__ __forceinline__ double shfl(double v, int src) { return __shfl_sync(0xffffffffu, v, src); }
__device__ __forceinline__ float2 shfl(float2 v, int src) {
    return make_float2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
}
__device__ __forceinline__ double2 shfl(double2 v, int src) {
    return make_double2(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src));
}

template <typename T, int M, int NC>
__global__ void __launch_bounds__(128) small_rowlane_kernel(const SmallGeom g, const T alpha) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int S = (M + 31) / 32;  // row slots per lane
    T *base = reinterpret_cast<T *>(smem_raw);
    const int per = SmallImage<T, M>::elems(NC);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    // blockIdx.y picks a slice of NC columns: a launch with gridDim.y > 1
    // spreads the columns of a few systems over many SMs
    const int j0 = blockIdx.y * NC;
    const int n = min(NC, g.n - j0);  // columns of this CTA
    const int64_t sys0 = (int64_t)blockIdx.x * g.spc;
    const int nsys = (int)min((int64_t)g.spc, g.batch - sys0);

    for (int s = 0; s < nsys; ++s) {
        T *Ls = base + s * per;
        stage_system<T, M>(g, Ls, Ls + SmallImage<T, M>::kLs, Ls + SmallImage<T, M>::kLs + M, sys0 + s, j0, n,
                           tid, nthr);
    }
    cp_async_wait_all();
    __syncthreads();

    if (warp < nsys) {  // warp-uniform
        const T *Ls = base + warp * per;
        const T *dinv = Ls + SmallImage<T, M>::kLs;
        T *Bs = base + warp * per + SmallImage<T, M>::kLs + M;
        T b[S][NC];
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            const int i = lane + 32 * s2;
#pragma unroll
            for (int c = 0; c < NC; ++c)
                b[s2][c] = (i < M && c < n) ? mul(alpha, Bs[c * (M + 1) + i]) : zero_of<T>();
        }
#pragma unroll
        for (int k = 0; k < M; ++k) {
            const int owner = k & 31, slot = k >> 5;
            const T d = dinv[k];
            T x[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) x[c] = mul(shfl(b[slot][c], owner), d);
            if (lane == owner) {
#pragma unroll
                for (int c = 0; c < NC; ++c) b[slot][c] = x[c];
            }
#pragma unroll
            for (int s2 = slot; s2 < S; ++s2) {
                const int i = lane + 32 * s2;
                if (i > k && i < M) {
                    const T l = Packed<T, M>::col(Ls, k)[i];
#pragma unroll
                    for (int c = 0; c < NC; ++c) b[s2][c] = fms(l, x[c], b[s2][c]);
                }
            }
        }
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            const int i = lane + 32 * s2;
#pragma unroll
            for (int c = 0; c < NC; ++c)
                if (i < M && c < n) Bs[c * (M + 1) + i] = b[s2][c];
        }
    }
    __syncthreads();

    for (int q = 0; q < nsys; ++q)
        unstage_system<T, M>(g, base + q * per + SmallImage<T, M>::kLs + M, sys0 + q, j0, n, tid, nthr);
}

// ---------------------------------------------------------------- alpha == 0
// B <- 0 for every system, without reading A (BLAS convention).
template <typename T>
__global__ void zero_rhs_kernel(T *B, int64_t rows, int64_t cols, int64_t ld, int64_t stride, int64_t batch,
                                int layout) {
    const int64_t per = rows * cols;
    const int64_t total = per * batch;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = e / per, r = e - b * per;
        int64_t off;
        if (layout == 0) off = (r / rows) * ld + (r % rows);  // column-major: r = j*rows + i
        else off = (r / cols) * ld + (r % cols);              // row-major:    r = i*cols + j
        B[b * stride + off] = zero_of<T>();
    }
}

}  // namespace trsm
