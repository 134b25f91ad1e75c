// Kernels of the blocked (m > 64) path.
//
// "Hierarchical Shared Memory-Aware Optimization for TRSM on GPU Platforms":
// the lower triangle is split into block rows of NB; every diagonal block D_t
// is inverted independently (different D_t go to different CTAs), each D_t
// itself in I_B x I_B sub-blocks with I_B = NB/8.  The diagonal sub-blocks
// are inverted by pure column-level substitution against identity tiles,
// loading one column at a time into a double buffer (O(I_B) shared memory);
// the inter-sub-block terms become matrix products through the blocked
// triangular-inverse formula.  The solve then applies D_t^{-1} to the block
// row and updates the trailing right-hand side with a GEMM, the dominant cost.
#pragma once

#include "common.cuh"
#include "small_kernels.cuh"  // Vec, lds16, update_rows

namespace trsm {

// ---------------------------------------------------------------------------
// Level 1: invert the diagonal I_B x I_B sub-block S of D_t.
// CTA (t, i) handles S = L[r0 : r0+IB, r0 : r0+IB], r0 = t*NB + i*IB.
// Thread j solves S y = e_j (column j of the identity tile) with y in
// registers.  Column k of S is streamed through a two-slot shared buffer:
// while slot k&1 feeds step k, slot (k+1)&1 receives column k+1 by cp.async.
// Rows and columns at or beyond m are identity padding.
// Output: the lower triangle of S^{-1} into W_t (NB x NB, column-major, ld
// NB) at sub-block (i, i); the strictly upper sub-blocks (0..i-1, i) of
// column block i are zero-filled.
// ---------------------------------------------------------------------------
template <typename T, int IB>
__device__ __forceinline__ void inv_l1_prefetch(T *slot, const T *L, int64_t lda, int64_t m, int64_t r0, int k,
                                                int tid) {
    // rows 0..IB-1 of column k; thread tid loads row tid (IB threads)
    const int64_t gr = r0 + tid, gc = r0 + k;
    if (tid > k && gr < m) cp_async<sizeof(T)>(slot + tid, L + gc * lda + gr);
    else if (tid == k) slot[tid] = (gr < m) ? ldg(L + gc * lda + gr) : T{};
    else slot[tid] = zero_of<T>();
}


template <typename T, int IB, int K>
struct InvL1Steps {
    static __device__ __forceinline__ void run(T (&y)[IB], T (*buf)[IB], const T *L, int64_t lda, int64_t m,
                                               int64_t r0, int tid) {
        if constexpr (K < IB) {
            if (K + 1 < IB) inv_l1_prefetch<T, IB>(buf[(K + 1) & 1], L, lda, m, r0, K + 1, tid);
            cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            const T *col = buf[K & 1];
            const T d = (r0 + K < m) ? col[K] : one_of<T>();
            const T xk = mul(y[K], recip(d));
            y[K] = xk;
            update_rows<T, IB, K + 1>(col, xk, y);
            __syncthreads();
            InvL1Steps<T, IB, K + 1>::run(y, buf, L, lda, m, r0, tid);
        }
    }
};

template <typename T, int IB>
__global__ void __launch_bounds__(IB) inv_diag_l1_kernel(const T *__restrict__ L, int64_t lda, int64_t m, int nb,
                                                         T *__restrict__ W, int64_t sL = 0, int64_t sW = 0) {
    // grid y: systems of a batch (L and W advance by sL / sW elements)
    L += (int64_t)blockIdx.y * sL;
    W += (int64_t)blockIdx.y * sW;
    __shared__ __align__(16) T buf[2][IB];
    const int t = blockIdx.x / 8, i = blockIdx.x % 8;
    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)t * nb + (int64_t)i * IB;
    T y[IB];
#pragma unroll
    for (int r = 0; r < IB; ++r) y[r] = (r == tid) ? one_of<T>() : zero_of<T>();
    inv_l1_prefetch<T, IB>(buf[0], L, lda, m, r0, 0, tid);
    cp_async_commit();
    InvL1Steps<T, IB, 0>::run(y, buf, L, lda, m, r0, tid);
    cp_async_wait_all();

    T *Wt = W + (int64_t)t * nb * nb;
    const int c = i * IB + tid;  // column of W_t owned by this thread
    T *colp = Wt + (int64_t)c * nb;
    for (int r = 0; r < i * IB; ++r) colp[r] = zero_of<T>();
#pragma unroll
    for (int r = 0; r < IB; ++r) colp[i * IB + r] = y[r];
}

// ---------------------------------------------------------------------------
// Level 2: off-diagonal sub-blocks of W_t = D_t^{-1}.  With S_ii the
// diagonal sub-blocks and L_ik the sub-blocks of D_t,
//     Y_ij = -Y_ii * sum_{k=j}^{i-1} L_ik Y_kj ,
// every Y_kj on the right lying in the same block column j, above row
// block i.  CTA (t, j) therefore walks down its block column, i = j+1 .. 7,
// in one launch: for each i it forms P = L[i-rows, j..i-1 cols] *
// Y[j..i-1 rows, j col] (K = (i-j)*IB) in shared memory, then
// Y_ij = -Y_ii * P, and a block barrier publishes Y_ij to the next i.
// 256 threads, each owning a TR x TC patch.
// ---------------------------------------------------------------------------
template <typename T, int IB>
struct L2Cfg {
    static constexpr int kThreads = 256;
    static constexpr int kTR = IB >= 64 ? 4 : (IB >= 32 ? 2 : 1);
    static constexpr int kTC = IB >= 64 ? 4 : (IB >= 32 ? 2 : 1);
    static constexpr int kKC = 16;  // K chunk staged per step
    static_assert((IB / kTR) * (IB / kTC) == kThreads, "level-2 thread tiling");
};

template <typename T, int IB>
__device__ __forceinline__ void inv_offdiag_block(const T *__restrict__ L, int64_t lda, int64_t m, int nb,
                                                  T *__restrict__ W, int d) {
    using C = L2Cfg<T, IB>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T *La = reinterpret_cast<T *>(smem_raw);  // [KC][IB]  (k-major chunk of L rows)
    T *Yb = La + C::kKC * IB;                 // [KC][IB]  (k-major chunk of Y_kj)
    T *P = Yb + C::kKC * IB;                  // [IB][IB + 1] column-major, padded
    T *Yd = P + IB * (IB + 1);                // [IB][IB + 1] Y_ii column-major, padded
    const int t = blockIdx.x, j = blockIdx.y, i = j + d;
    const int tid = threadIdx.x;
    const int tr = tid % (IB / C::kTR), tc = tid / (IB / C::kTR);
    T *Wt = W + (int64_t)t * nb * nb;
    const int64_t grow0 = (int64_t)t * nb + (int64_t)i * IB;   // global row of sub-block row i
    const int64_t gcol0 = (int64_t)t * nb + (int64_t)j * IB;   // global col of sub-block col j
    const int K = d * IB;

    T acc[C::kTR][C::kTC];
#pragma unroll
    for (int a = 0; a < C::kTR; ++a)
#pragma unroll
        for (int b = 0; b < C::kTC; ++b) acc[a][b] = zero_of<T>();

    for (int k0 = 0; k0 < K; k0 += C::kKC) {
        __syncthreads();
        for (int e = tid; e < C::kKC * IB; e += C::kThreads) {
            const int kk = e / IB, r = e % IB;
            const int64_t gr = grow0 + r, gc = gcol0 + k0 + kk;
            La[kk * IB + r] = (gr < m) ? ldg(L + gc * lda + gr) : zero_of<T>();
        }
        for (int e = tid; e < C::kKC * IB; e += C::kThreads) {
            const int kk = e % C::kKC, c = e / C::kKC;
            // Y_kj rows j*IB + k0 + kk (contiguous in W_t), column j*IB + c
            Yb[kk * IB + c] = Wt[(int64_t)(j * IB + c) * nb + (j * IB + k0 + kk)];
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < C::kKC; ++kk) {
            T a[C::kTR], b[C::kTC];
#pragma unroll
            for (int q = 0; q < C::kTR; ++q) a[q] = La[kk * IB + tr * C::kTR + q];
#pragma unroll
            for (int q = 0; q < C::kTC; ++q) b[q] = Yb[kk * IB + tc * C::kTC + q];
#pragma unroll
            for (int x = 0; x < C::kTR; ++x)
#pragma unroll
                for (int y = 0; y < C::kTC; ++y) acc[x][y] = fma_(a[x], b[y], acc[x][y]);
        }
    }
    // P and Y_ii into shared memory
#pragma unroll
    for (int x = 0; x < C::kTR; ++x)
#pragma unroll
        for (int y = 0; y < C::kTC; ++y) P[(tc * C::kTC + y) * (IB + 1) + tr * C::kTR + x] = acc[x][y];
    for (int e = tid; e < IB * IB; e += C::kThreads) {
        const int c = e / IB, r = e % IB;
        Yd[c * (IB + 1) + r] = Wt[(int64_t)(i * IB + c) * nb + (i * IB + r)];
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < C::kTR; ++a)
#pragma unroll
        for (int b = 0; b < C::kTC; ++b) acc[a][b] = zero_of<T>();
    for (int k = 0; k < IB; ++k) {
        T a[C::kTR], b[C::kTC];
#pragma unroll
        for (int q = 0; q < C::kTR; ++q) a[q] = Yd[k * (IB + 1) + tr * C::kTR + q];
#pragma unroll
        for (int q = 0; q < C::kTC; ++q) b[q] = P[(tc * C::kTC + q) * (IB + 1) + k];
#pragma unroll
        for (int x = 0; x < C::kTR; ++x)
#pragma unroll
            for (int y = 0; y < C::kTC; ++y) acc[x][y] = fms(a[x], b[y], acc[x][y]);
    }
    // Y_ij into W_t rows i*IB.., cols j*IB..
#pragma unroll
    for (int y = 0; y < C::kTC; ++y) {
        T *colp = Wt + (int64_t)(j * IB + tc * C::kTC + y) * nb + i * IB + tr * C::kTR;
#pragma unroll
        for (int x = 0; x < C::kTR; ++x) colp[x] = acc[x][y];
    }
}

template <typename T, int IB>
__global__ void __launch_bounds__(256) inv_offdiag_kernel(const T *__restrict__ L, int64_t lda, int64_t m, int nb,
                                                          T *__restrict__ W, int64_t sL = 0, int64_t sW = 0) {
    // grid z: systems of a batch
    L += (int64_t)blockIdx.z * sL;
    W += (int64_t)blockIdx.z * sW;
    for (int d = 1; d < 8 - (int)blockIdx.y; ++d) {
        inv_offdiag_block<T, IB>(L, lda, m, nb, W, d);
        __syncthreads();  // Y_ij is read by the next sub-block of this column
    }
}

template <typename T, int IB>
constexpr size_t inv_offdiag_smem() {
    return sizeof(T) * (2 * L2Cfg<T, IB>::kKC * IB + 2 * IB * (IB + 1));
}

// ---------------------------------------------------------------------------
// One CTA (256 threads) inverts a whole 128 x 128 diagonal block D_t in
// shared memory, for the few-right-hand-side path: the two kernels above
// (sub-blocks in CTAs of I_B threads, then the off-diagonal sub-blocks one
// after another) are latency-bound at NB = 128.  The same blocked
// triangular-inverse formula, level by level, in place:
//   level 1  warps 0-3 invert the four 32 x 32 diagonal sub-blocks by
//            substitution against identity columns (lane j: column j, in
//            registers, column k of the sub-block read as a broadcast);
//   level 2  each 64 x 64 diagonal block [[A, 0], [C, B]], A^{-1} and B^{-1}
//            known, gets its lower-left block -B^{-1} (C A^{-1}): two
//            products, the middle one in a temporary;
//   level 3  the same for the whole block with 64 x 64 parts.
// The products skip the zero triangles of A^{-1} and B^{-1}.  Rows and
// columns at or beyond m are identity padding; the strictly upper triangle
// is zero.  Output W_t: 128 x 128, column-major, ld 128, at W + t 128^2.
// Used for f32 and c64 (the block and a 64 x 64 temporary fit the 227 KB
// up to 8-byte elements; in f64 one SM's FP64 rate makes the two-kernel
// inversion, spread over more CTAs, the faster one).
// ---------------------------------------------------------------------------
constexpr int kInvN = 128, kInvLd = kInvN + 1, kInvTmpLd = 65;

template <typename T>
constexpr size_t inv_block128_smem() {
    return sizeof(T) * ((size_t)kInvN * kInvLd + (size_t)64 * kInvTmpLd);
}

// C = (NEG ? -1 : 1) A B over R x R parts (column-major, leading dimensions
// la, lb, lc); A lower triangular when A_LOWER, B when B_LOWER.  Thread lt of
// the (R/PR)(R/PC) taking part owns rows i0 .. i0+PR-1, columns j0 .. j0+PC-1.
template <typename T, int R, int PR, int PC, bool A_LOWER, bool B_LOWER, bool NEG>
__device__ __forceinline__ void inv_part_product(const T *A, int la, const T *Bm, int lb, T *Cm, int lc, int lt) {
    const int i0 = (lt % (R / PR)) * PR, j0 = (lt / (R / PR)) * PC;
    T acc[PR][PC];
#pragma unroll
    for (int x = 0; x < PR; ++x)
#pragma unroll
        for (int y = 0; y < PC; ++y) acc[x][y] = zero_of<T>();
    const int k_lo = B_LOWER ? j0 : 0;               // B(k, j) = 0 for k < j
    const int k_hi = A_LOWER ? i0 + PR : R;          // A(i, k) = 0 for k > i
#pragma unroll 2
    for (int k = k_lo; k < k_hi; ++k) {
        T a[PR], b[PC];
#pragma unroll
        for (int x = 0; x < PR; ++x) a[x] = A[k * la + i0 + x];
#pragma unroll
        for (int y = 0; y < PC; ++y) b[y] = Bm[(j0 + y) * lb + k];
#pragma unroll
        for (int x = 0; x < PR; ++x)
#pragma unroll
            for (int y = 0; y < PC; ++y) acc[x][y] = NEG ? fms(a[x], b[y], acc[x][y]) : fma_(a[x], b[y], acc[x][y]);
    }
#pragma unroll
    for (int x = 0; x < PR; ++x)
#pragma unroll
        for (int y = 0; y < PC; ++y) Cm[(j0 + y) * lc + i0 + x] = acc[x][y];
}

// CTA b inverts rows and columns b*128 .. of L.  With diagonal blocks of
// nbw = 128, 256 or 512 rows in W (ld nbw, one nbw^2 block after another),
// its inverse lands at sub-block (q, q) of W_t, t = b / (nbw/128),
// q = b % (nbw/128), and the rows above it in its columns are zeroed; the
// blocks below the 128-row diagonal come from invert_blocks_doubling.
// fill (optional): fill_words 32-bit words per CTA set to all ones, at
// fill + blockIdx.x fill_words (the few-right-hand-side path's published copy
// of X, cleared here instead of by a separate memset).
template <typename T>
__global__ void __launch_bounds__(256) inv_block128_kernel(const T *__restrict__ L, int64_t lda, int64_t m,
                                                           T *__restrict__ W, int nbw, uint32_t *__restrict__ fill,
                                                           int64_t fill_words) {
    extern __shared__ __align__(16) unsigned char inv_smem[];
    T *S = reinterpret_cast<T *>(inv_smem);  // D_t, then W_t: element (i, j) at j kInvLd + i
    T *Tmp = S + kInvN * kInvLd;             // 64 x 64 (or two 32 x 32), ld kInvTmpLd
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t r0 = (int64_t)blockIdx.x * kInvN;
    const int mb = (int)(m - r0 < kInvN ? m - r0 : kInvN);
    {
        // thread: row i of columns j0, j0 + 2, ..., 32 loads in flight at a time
        const int i = tid % kInvN, j0 = tid / kInvN;
#pragma unroll 1
        for (int q0 = 0; q0 < kInvN / 2; q0 += 32) {
            T v[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int j = j0 + 2 * (q0 + q);
                v[q] = (i >= j && i < mb) ? L[(r0 + j) * lda + r0 + i] : (i == j ? one_of<T>() : zero_of<T>());
            }
#pragma unroll
            for (int q = 0; q < 32; ++q) S[(j0 + 2 * (q0 + q)) * kInvLd + i] = v[q];
        }
    }
    __syncthreads();
    if (warp < 4) {
        // level 1: lane j solves D_ww y = e_j for the sub-block at rows and
        // columns 32 warp ..; right-looking, y_k final at step k
        T *D = S + warp * 32 * (kInvLd + 1);
        T y[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = i == lane ? one_of<T>() : zero_of<T>();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const T *col = D + k * kInvLd;
            y[k] = mul(y[k], recip(col[k]));
#pragma unroll
            for (int i = k + 1; i < 32; ++i) y[i] = fms(col[i], y[k], y[i]);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) D[lane * kInvLd + i] = y[i];
    }
    __syncthreads();
    {
        // level 2: the two 64 x 64 diagonal blocks at o = 0, 64, 128 threads each
        const int o = (tid >> 7) * 64, lt = tid & 127;
        T *A = S + o * kInvLd + o, *Bi = S + (o + 32) * kInvLd + o + 32, *C = S + o * kInvLd + o + 32;
        T *P = Tmp + (tid >> 7) * 32 * kInvTmpLd;
        inv_part_product<T, 32, 4, 2, false, true, false>(C, kInvLd, A, kInvLd, P, kInvTmpLd, lt);
        __syncthreads();
        inv_part_product<T, 32, 4, 2, true, false, true>(Bi, kInvLd, P, kInvTmpLd, C, kInvLd, lt);
        __syncthreads();
    }
    {
        // level 3: the whole block, 64 x 64 parts
        T *A = S, *Bi = S + 64 * kInvLd + 64, *C = S + 64;
        inv_part_product<T, 64, 4, 4, false, true, false>(C, kInvLd, A, kInvLd, Tmp, kInvTmpLd, tid);
        __syncthreads();
        inv_part_product<T, 64, 4, 4, true, false, true>(Bi, kInvLd, Tmp, kInvTmpLd, C, kInvLd, tid);
        __syncthreads();
    }
    const int per = nbw / kInvN, q = (int)(blockIdx.x % per);
    T *Wt = W + (int64_t)(blockIdx.x / per) * nbw * nbw + (int64_t)q * kInvN * (nbw + 1);
    for (int e = tid; e < kInvN * kInvN; e += 256) Wt[(e / kInvN) * nbw + e % kInvN] = S[(e / kInvN) * kInvLd + e % kInvN];
    for (int e = tid; e < q * kInvN * kInvN; e += 256) {
        const int i = e % (q * kInvN), j = e / (q * kInvN);
        Wt[(int64_t)j * nbw + i - q * kInvN] = zero_of<T>();
    }
    if (fill)
        for (int64_t e = tid; e < fill_words; e += 256) fill[(int64_t)blockIdx.x * fill_words + e] = 0xffffffffu;
}

// ---------------------------------------------------------------------------
// Tiled GEMM  C = beta*C + gamma * A * B  (all column-major; beta_zero skips
// reading C).  With a_lower, A is lower triangular and the K loop of a
// row tile stops at the tile's last row.  256 threads, a TM x TN register
// patch per thread, double-buffered cp.async staging of BK-deep slabs.
// ---------------------------------------------------------------------------
template <typename T, bool SMALL> struct GemmCfg;
template <> struct GemmCfg<float, false>   { static constexpr int BM = 128, BN = 128, BK = 16, TM = 8, TN = 8; };
template <> struct GemmCfg<double, false>  { static constexpr int BM = 64,  BN = 64,  BK = 16, TM = 4, TN = 4; };
template <> struct GemmCfg<float2, false>  { static constexpr int BM = 64,  BN = 64,  BK = 16, TM = 4, TN = 4; };
template <> struct GemmCfg<double2, false> { static constexpr int BM = 64,  BN = 32,  BK = 8,  TM = 4, TN = 2; };
// small tiles: 4x more CTAs for grids below two waves
template <> struct GemmCfg<float, true>    { static constexpr int BM = 64,  BN = 64,  BK = 16, TM = 4, TN = 4; };
template <> struct GemmCfg<double, true>   { static constexpr int BM = 32,  BN = 32,  BK = 16, TM = 2, TN = 2; };
template <> struct GemmCfg<float2, true>   { static constexpr int BM = 32,  BN = 32,  BK = 16, TM = 2, TN = 2; };
template <> struct GemmCfg<double2, true>  { static constexpr int BM = 32,  BN = 16,  BK = 8,  TM = 2, TN = 1; };

template <typename T>
struct GemmArgs {
    int64_t M, N, K;
    const T *A;
    int64_t lda;
    const T *B;
    int64_t ldb;
    T *C;
    int64_t ldc;
    T gamma, beta;
    int beta_zero, a_lower;
    int b_rowmajor;  // B element (k, c) at k*ldb + c instead of c*ldb + k
    int c_rowmajor;  // C element (r, c) at r*ldc + c instead of c*ldc + r
    int64_t sA = 0, sB = 0, sC = 0;  // grid z: systems of a batch, element strides
};

template <typename T, bool SMALL>
__global__ void __launch_bounds__(256) gemm_kernel(const GemmArgs<T> g) {
    using C = GemmCfg<T, SMALL>;
    constexpr int BM = C::BM, BN = C::BN, BK = C::BK, TM = C::TM, TN = C::TN;
    constexpr int NT = (BM / TM) * (BN / TN);
    static_assert(NT == 256, "gemm threads");
    constexpr int BPAD = 16 / (int)sizeof(T) > 1 ? 16 / (int)sizeof(T) : 1;
    __shared__ __align__(16) T As[2][BK][BM];
    __shared__ __align__(16) T Bs[2][BK][BN + BPAD];

    const int tid = threadIdx.x;
    const int tx = tid % (BM / TM), ty = tid / (BM / TM);
    const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
    const T *gA = g.A + (int64_t)blockIdx.z * g.sA;
    const T *gB = g.B + (int64_t)blockIdx.z * g.sB;
    T *gC = g.C + (int64_t)blockIdx.z * g.sC;
    int64_t kend = g.K;
    if (g.a_lower && m0 + BM < kend) kend = m0 + BM;
    const int nk = (int)((kend + BK - 1) / BK);

    auto load = [&](int kt, int s) {
        const int64_t k0 = (int64_t)kt * BK;
        for (int e = tid; e < BM * BK; e += NT) {
            const int kk = e / BM, r = e % BM;
            const int64_t gr = m0 + r, gk = k0 + kk;
            if (gr < g.M && gk < kend) cp_async<sizeof(T)>(&As[s][kk][r], gA + gk * g.lda + gr);
            else As[s][kk][r] = zero_of<T>();
        }
        if (g.b_rowmajor) {
            for (int e = tid; e < BK * BN; e += NT) {
                const int kk = e / BN, c = e % BN;
                const int64_t gc = n0 + c, gk = k0 + kk;
                if (gc < g.N && gk < kend) cp_async<sizeof(T)>(&Bs[s][kk][c], gB + gk * g.ldb + gc);
                else Bs[s][kk][c] = zero_of<T>();
            }
        } else {
            for (int e = tid; e < BK * BN; e += NT) {
                const int kk = e % BK, c = e / BK;
                const int64_t gc = n0 + c, gk = k0 + kk;
                if (gc < g.N && gk < kend) cp_async<sizeof(T)>(&Bs[s][kk][c], gB + gc * g.ldb + gk);
                else Bs[s][kk][c] = zero_of<T>();
            }
        }
    };

    T acc[TM][TN];
#pragma unroll
    for (int a = 0; a < TM; ++a)
#pragma unroll
        for (int b = 0; b < TN; ++b) acc[a][b] = zero_of<T>();

    if (nk > 0) load(0, 0);
    cp_async_commit();
    for (int kt = 0; kt < nk; ++kt) {
        if (kt + 1 < nk) load(kt + 1, (kt + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const int s = kt & 1;
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            T a[TM], b[TN];
#pragma unroll
            for (int q = 0; q < TM; ++q) a[q] = As[s][kk][tx * TM + q];
#pragma unroll
            for (int q = 0; q < TN; ++q) b[q] = Bs[s][kk][ty * TN + q];
#pragma unroll
            for (int x = 0; x < TM; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) acc[x][y] = fma_(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
    }
    cp_async_wait_all();

#pragma unroll
    for (int y = 0; y < TN; ++y) {
        const int64_t gc = n0 + ty * TN + y;
        if (gc >= g.N) continue;
#pragma unroll
        for (int x = 0; x < TM; ++x) {
            const int64_t gr = m0 + tx * TM + x;
            if (gr >= g.M) continue;
            T *cp = g.c_rowmajor ? gC + gr * g.ldc + gc : gC + gc * g.ldc + gr;
            T v = mul(g.gamma, acc[x][y]);
            if (!g.beta_zero) v = fma_(g.beta, *cp, v);
            *cp = v;
        }
    }
}

// dst (column-major rows x cols, ld_dst) = transpose-view of src, where src
// holds the same logical matrix row-major (ld_src): dst[c*ld_dst + r] =
// src[r*ld_src + c].  32 x 32 tiles through shared memory.
template <typename T>
__global__ void transpose_kernel(const T *__restrict__ src, int64_t ld_src, T *__restrict__ dst, int64_t ld_dst,
                                 int64_t rows, int64_t cols, int64_t s_src = 0, int64_t s_dst = 0) {
    // grid z: systems of a batch
    src += (int64_t)blockIdx.z * s_src;
    dst += (int64_t)blockIdx.z * s_dst;
    __shared__ T tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.y * 32, c0 = (int64_t)blockIdx.x * 32;
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + q, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[q][threadIdx.x] = src[r * ld_src + c];
    }
    __syncthreads();
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t c = c0 + q, r = r0 + threadIdx.x;
        if (r < rows && c < cols) dst[c * ld_dst + r] = tile[threadIdx.x][q];
    }
}

}  // namespace trsm
