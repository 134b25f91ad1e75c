// Persistent complex64 small-regime kernel on the TMA engine (m = 32, 48,
// 64): the f32 kernel's design (small_fast.cuh) carried over to complex
// arithmetic on paired FP32 FMAs.
//
// Work: items (system, W-column slice of the right-hand side), W = 64 (a
// pair of warps per item) or 32 (one warp); one column per thread, kept in
// registers 16 rows at a time.  Each unit of W threads streams its own
// sequence of items through a two-stage shared-memory ring:
//   in   the lower 16 x 16 complex blocks of L as tiled tensor copies (128
//        bytes = 16 complex rows per line, one line per column), and the
//        right-hand-side slice as 16-row x W-column boxes with the 128-byte
//        swizzle (16-byte chunk q of line c at chunk q ^ (c % 8)), so a
//        thread reading its own column meets no bank conflicts;
//   out  X is written back over its right-hand-side column and leaves as the
//        same boxes (the tensor store clips columns past n).
// On arrival every line of L is rewritten in place from interleaved
// (re, im) pairs into planar form -- the 16 real parts, then the 16
// imaginary parts -- so that one 16-byte shared load yields the real (or
// imaginary) parts of four consecutive rows.  The solve then keeps each row
// pair's real parts and imaginary parts in two 64-bit registers and updates
// them with four fma.rn.f32x2 per pair and column of L:
//     re -= Re L * Re x ;  re += Im L * Im x ;
//     im -= Re L * Im x ;  im -= Im L * Re x .
// Rows of earlier 16-row chunks are read back from the stage (the solved
// rows are written there), so the loop over them stays rolled and the code
// small enough for the instruction cache.
#pragma once

#include "internal.h"
#include "mbarrier.cuh"
#include "small_fast.cuh"

namespace trsm {

template <int M, int W>
struct C64Stage {
    static_assert(M == 32 || M == 48 || M == 64, "16-row blocks, m >= 32");
    static_assert(W == 32 || W == 64, "column slice");
    static constexpr int NR = M / 16;                         // 16-row blocks
    static constexpr int kLBoxes = NR * (NR + 1) / 2;         // lower blocks of L
    static constexpr int kLFloats = kLBoxes * 512;            // 2 KB per block
    static constexpr int kBBox = W * 32;                      // floats per RHS box
    static constexpr int kBFloats = NR * kBBox;
    static constexpr int kDFloats = 256;                      // 1 KB: M reciprocals (re, im), padded
    static constexpr int kElems = kLFloats + kBFloats + kDFloats;
    static constexpr uint32_t kLoadBytes = 4u * (kLFloats + kBFloats);
    static_assert(kLFloats % 256 == 0 && kBBox % 256 == 0 && kElems % 256 == 0, "1024-byte aligned regions");
    static_assert(2 * M <= kDFloats, "reciprocals");
    // block (rb, cb) of L (rows 16 rb.., columns 16 cb..), rb >= cb
    static __host__ __device__ constexpr int lbox(int rb, int cb) { return (rb * (rb + 1) / 2 + cb) * 512; }
    static __host__ __device__ constexpr int bbox(int rb) { return kLFloats + rb * kBBox; }
    static __host__ __device__ constexpr int dinv() { return kLFloats + kBFloats; }
};

// ST stages per unit (2: the next item's copies overlap this item's solve;
// 1: a unit waits for its own copies, and twice as many units share the SM
// -- more warps to hide each other's latencies), as many units as fit.
template <int M, int W, int ST>
struct C64Units {
    using S = C64Stage<M, W>;
    static_assert(ST == 1 || ST == 2, "stages");
    static constexpr int kStageBytes = 4 * S::kElems;
    static constexpr int kFit = (226 * 1024) / (ST * kStageBytes);
    static constexpr int kMaxUnits = 8 / (W / 32);  // at most 8 warps (255 registers a thread)
    static constexpr int kUnits = kFit > kMaxUnits ? kMaxUnits : kFit;
    static_assert(kUnits >= 1, "stages per unit");
    static constexpr int kThreads = W * kUnits;
    static constexpr size_t kSmem = (size_t)kUnits * ST * kStageBytes + 1024;
};

__device__ __forceinline__ f32x2 dup2(float v) { return pack2(v, v); }

// Step kk of the diagonal block of chunk R (rows 16R..16R+15): x = b_kk /
// L_kk, then the rows below kk within the chunk.
template <int KK>
struct C64Diag {
    static __device__ __forceinline__ void run(const float *__restrict__ lcol0, const float *__restrict__ dinv,
                                               f32x2 (&br)[8], f32x2 (&bi)[8]) {
        if constexpr (KK < 16) {
            constexpr int pk = KK / 2, half = KK % 2;
            const float *lcol = lcol0 + KK * 32;  // planar line of column KK: re[16], im[16]
            const float2 d = *reinterpret_cast<const float2 *>(dinv + 2 * KK);
            float r0, r1, i0, i1;
            unpack2(br[pk], r0, r1);
            unpack2(bi[pk], i0, i1);
            const float bre = half ? r1 : r0, bim = half ? i1 : i0;
            const float xre = bre * d.x - bim * d.y;
            const float xim = bre * d.y + bim * d.x;
            if constexpr (half == 0) {
                // the partner row KK+1 of the same pair
                const float lre = lcol[KK + 1], lim = lcol[16 + KK + 1];
                r1 = fmaf(-lre, xre, fmaf(lim, xim, r1));
                i1 = fmaf(-lre, xim, fmaf(-lim, xre, i1));
                r0 = xre;
                i0 = xim;
            } else {
                r1 = xre;
                i1 = xim;
            }
            br[pk] = pack2(r0, r1);
            bi[pk] = pack2(i0, i1);
            const f32x2 nxr = dup2(-xre), pxi = dup2(xim), nxi = dup2(-xim);
#pragma unroll
            for (int p = pk + 1; p < 8; ++p) {
                const f32x2 lr = *reinterpret_cast<const f32x2 *>(lcol + 2 * p);
                const f32x2 li = *reinterpret_cast<const f32x2 *>(lcol + 16 + 2 * p);
                br[p] = ffma2(lr, nxr, br[p]);
                br[p] = ffma2(li, pxi, br[p]);
                bi[p] = ffma2(lr, nxi, bi[p]);
                bi[p] = ffma2(li, nxr, bi[p]);
            }
            C64Diag<KK + 1>::run(lcol0, dinv, br, bi);
        }
    }
};

// Two earlier columns k, k+1 (x = (x.x, x.y) and (x.z, x.w)) into the 16
// rows of the chunk: lcol is the planar line of column k (rows 16R..16R+15),
// lcol + 32 that of column k+1.  Every load is issued first, then the 64
// paired FMAs in four sweeps over the 16 accumulators, so that consecutive
// FMAs on one accumulator are 16 instructions apart.
__device__ __forceinline__ void c64_col_update2(const float *__restrict__ lcol, const float4 x, f32x2 (&br)[8],
                                                f32x2 (&bi)[8]) {
    ulonglong2 lr0[4], li0[4], lr1[4], li1[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        lr0[q] = *reinterpret_cast<const ulonglong2 *>(lcol + 4 * q);
        li0[q] = *reinterpret_cast<const ulonglong2 *>(lcol + 16 + 4 * q);
        lr1[q] = *reinterpret_cast<const ulonglong2 *>(lcol + 32 + 4 * q);
        li1[q] = *reinterpret_cast<const ulonglong2 *>(lcol + 48 + 4 * q);
    }
    const f32x2 nxr0 = dup2(-x.x), pxi0 = dup2(x.y), nxi0 = dup2(-x.y);
    const f32x2 nxr1 = dup2(-x.z), pxi1 = dup2(x.w), nxi1 = dup2(-x.w);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        br[2 * q] = ffma2(lr0[q].x, nxr0, br[2 * q]);
        br[2 * q + 1] = ffma2(lr0[q].y, nxr0, br[2 * q + 1]);
        bi[2 * q] = ffma2(lr0[q].x, nxi0, bi[2 * q]);
        bi[2 * q + 1] = ffma2(lr0[q].y, nxi0, bi[2 * q + 1]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        br[2 * q] = ffma2(li0[q].x, pxi0, br[2 * q]);
        br[2 * q + 1] = ffma2(li0[q].y, pxi0, br[2 * q + 1]);
        bi[2 * q] = ffma2(li0[q].x, nxr0, bi[2 * q]);
        bi[2 * q + 1] = ffma2(li0[q].y, nxr0, bi[2 * q + 1]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        br[2 * q] = ffma2(lr1[q].x, nxr1, br[2 * q]);
        br[2 * q + 1] = ffma2(lr1[q].y, nxr1, br[2 * q + 1]);
        bi[2 * q] = ffma2(lr1[q].x, nxi1, bi[2 * q]);
        bi[2 * q + 1] = ffma2(lr1[q].y, nxi1, bi[2 * q + 1]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        br[2 * q] = ffma2(li1[q].x, pxi1, br[2 * q]);
        br[2 * q + 1] = ffma2(li1[q].y, pxi1, br[2 * q + 1]);
        bi[2 * q] = ffma2(li1[q].x, nxr1, bi[2 * q]);
        bi[2 * q + 1] = ffma2(li1[q].y, nxr1, bi[2 * q + 1]);
    }
}

template <int M, int W, int ST>
__global__ void __launch_bounds__(C64Units<M, W, ST>::kThreads, 1)
    small_tma_c64_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                         const int n, const float2 alpha, const int64_t items, int *status) {
    static_assert(ST == 1, "one region per unit, refilled chunk by chunk");
    using S = C64Stage<M, W>;
    constexpr int NR = S::NR, UNITS = C64Units<M, W, ST>::kUnits, UT = W;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // per unit and 16-row block J: barL[J] = column block J of L (blocks
    // (J..NR-1, J)), barB[J] = right-hand-side box J; each completes once per item
    __shared__ __align__(8) uint64_t barL[UNITS][NR], barB[UNITS][NR];
    const int tid = threadIdx.x;
    const int unit = tid / UT, pt = tid % UT;  // pt: this thread's column of the slice
    const bool leader = pt == 0;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;  // the swizzle pattern repeats every 1024 bytes
    float *cur = reinterpret_cast<float *>(smem_raw + (sbase - raw)) + unit * S::kElems;
    float *dinv = cur + S::dinv();
    if (tid < UNITS * NR) {
        mbar_init(smem_u32(&barL[tid / NR][tid % NR]), 1);
        mbar_init(smem_u32(&barB[tid / NR][tid % NR]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    __syncthreads();

    const int slices = (n + W - 1) / W;
    auto coords = [&](int64_t item, int &sys, int &j0) {
        sys = (int)(item / slices);
        j0 = (int)(item - (int64_t)sys * slices) * W;
    };
    // the unit's leader: column block J of L, and right-hand-side box J
    auto issue_l = [&](int64_t item, int J) {
        int sys, j0;
        coords(item, sys, j0);
        const uint32_t bar = smem_u32(&barL[unit][J]);
        mbar_expect_tx(bar, (uint32_t)(NR - J) * 2048u);
        for (int rb = J; rb < NR; ++rb)
            tma_load_3d(smem_u32(cur + S::lbox(rb, J)), &mapA, 32 * rb, 16 * J, sys, bar);
    };
    auto issue_b = [&](int64_t item, int J) {
        int sys, j0;
        coords(item, sys, j0);
        const uint32_t bar = smem_u32(&barB[unit][J]);
        mbar_expect_tx(bar, (uint32_t)S::kBBox * 4u);
        tma_load_3d(smem_u32(cur + S::bbox(J)), &mapB, 32 * J, j0, sys, bar);
    };
    const bool alpha_one = alpha.x == 1.f && alpha.y == 0.f;
    const f32x2 ar = dup2(alpha.x), ai = dup2(alpha.y), nai = dup2(-alpha.y), one2 = dup2(1.f);
    // phases armed (leader) and observed (every thread) per barrier
    uint32_t armL[NR], armB[NR], seenL[NR], seenB[NR];
#pragma unroll
    for (int J = 0; J < NR; ++J) armL[J] = armB[J] = seenL[J] = seenB[J] = 0;

    int64_t item = (int64_t)blockIdx.x * UNITS + unit;
    const int64_t step = (int64_t)gridDim.x * UNITS;
    if (leader && item < items) {
#pragma unroll
        for (int J = 0; J < NR; ++J) {
            issue_l(item, J);
            issue_b(item, J);
            ++armL[J];
            ++armB[J];
        }
    }
    const int sw = pt & 7;
    bool failed = false;
    for (; item < items && !failed; item += step) {
        const bool more = item + step < items;
        // accumulators: chunk R collects -sum_J L_RJ X_J; alpha B_R joins it
        // when chunk R is solved, so box R is needed only from then on
        f32x2 br[NR][8], bi[NR][8];
#pragma unroll
        for (int R = 0; R < NR; ++R)
#pragma unroll
            for (int q = 0; q < 8; ++q) br[R][q] = bi[R][q] = 0ull;
#pragma unroll
        for (int J = 0; J < NR; ++J) {
            if (failed) continue;
            const bool okl = mbar_wait(smem_u32(&barL[unit][J]), seenL[J] & 1u);
            const bool okb = okl && mbar_wait(smem_u32(&barB[unit][J]), seenB[J] & 1u);
            if (unit_any(unit, UT, !okb)) {
                failed = true;
                continue;
            }
            ++seenL[J];
            ++seenB[J];
            // column block J of L to planar lines, in place (8 threads per line,
            // thread q holding complex rows 2q, 2q+1); the diagonal block's
            // reciprocals on the way
            for (int line = pt / 8; line < 16 * (NR - J); line += UT / 8) {
                const int q = pt % 8, rb = J + line / 16, c = line % 16;
                float *ln = cur + S::lbox(rb, J) + c * 32;
                const float4 v = *reinterpret_cast<const float4 *>(ln + 4 * q);
                __syncwarp();
                *reinterpret_cast<float2 *>(ln + 2 * q) = make_float2(v.x, v.z);
                *reinterpret_cast<float2 *>(ln + 16 + 2 * q) = make_float2(v.y, v.w);
                if (rb == J && (c >> 1) == q) {
                    const float2 dr = (c & 1) ? make_float2(v.z, v.w) : make_float2(v.x, v.y);
                    *reinterpret_cast<float2 *>(dinv + 2 * (16 * J + c)) = recip(dr);
                }
                __syncwarp();
            }
            unit_sync(unit, UT);
            // chunk J: alpha B_J + accumulated updates, then its diagonal block
            float *bcol = cur + S::bbox(J) + pt * 32;  // this thread's line of box J
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(bcol + 4 * (q ^ sw));
                const f32x2 r = pack2(v.x, v.z), i = pack2(v.y, v.w);
                if (alpha_one) {
                    br[J][q] = ffma2(r, one2, br[J][q]);
                    bi[J][q] = ffma2(i, one2, bi[J][q]);
                } else {
                    br[J][q] = ffma2(i, nai, ffma2(r, ar, br[J][q]));
                    bi[J][q] = ffma2(r, ai, ffma2(i, ar, bi[J][q]));
                }
            }
            C64Diag<0>::run(cur + S::lbox(J, J), dinv + 32 * J, br[J], bi[J]);
            // X chunk J over box J: it leaves from there, and feeds the updates
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float r0, r1, i0, i1;
                unpack2(br[J][q], r0, r1);
                unpack2(bi[J][q], i0, i1);
                *reinterpret_cast<float4 *>(bcol + 4 * (q ^ sw)) = make_float4(r0, i0, r1, i1);
            }
            fence_proxy_async_smem();
            unit_sync(unit, UT);
            if (leader) {
                int sys, j0;
                coords(item, sys, j0);
                tma_store_3d(&mapB, 32 * J, j0, sys, smem_u32(cur + S::bbox(J)));
                bulk_commit();
            }
            if (J + 1 < NR) {
#pragma unroll 1
                for (int k = 0; k < 16; k += 2) {
                    const float4 x = *reinterpret_cast<const float4 *>(bcol + 4 * ((k / 2) ^ sw));
#pragma unroll
                    for (int R = J + 1; R < NR; ++R)
                        c64_col_update2(cur + S::lbox(R, J) + k * 32, x, br[R], bi[R]);
                }
            }
            unit_sync(unit, UT);  // column block J and box J are read by every thread
            if (leader && more) {
                issue_l(item + step, J);  // the next item's column block J
                ++armL[J];
                if (J >= 1) {
                    bulk_wait_read<1>();  // the store of box J-1 has read it
                    issue_b(item + step, J - 1);
                    ++armB[J - 1];
                }
            }
        }
        if (!failed && leader && more) {
            bulk_wait_read<0>();
            issue_b(item + step, NR - 1);
            ++armB[NR - 1];
        }
    }
    if (failed) {
        // a copy never completed: report, let every copy in flight land, stop
        if (leader) {
            record_timeout(status);
#pragma unroll
            for (int J = 0; J < NR; ++J) {
                for (uint32_t p = seenL[J]; p < armL[J]; ++p) mbar_wait(smem_u32(&barL[unit][J]), p & 1u);
                for (uint32_t p = seenB[J]; p < armB[J]; ++p) mbar_wait(smem_u32(&barB[unit][J]), p & 1u);
            }
        }
    }
    if (leader) bulk_wait<0>();  // every store complete before the CTA's shared memory goes away
}

// The kernel when the shape and strides allow it (column-major, m in {32,
// 48, 64}, n > 16, base addresses, leading dimensions and batch strides
// 16-byte multiples, enough items to fill the GPU); kTmaNotApplicable
// otherwise.
template <int M, int W, int ST>
static int launch_tma_c64_mw(const SmallArgs &a, cudaStream_t st) {
    using U = C64Units<M, W, ST>;
    float2 alpha;
    memcpy(&alpha, a.alpha, sizeof(alpha));
    CUtensorMap ma, mb;
    // complex64 as float pairs: dimension 0 runs over 2m floats of a column
    const uint64_t da[3] = {(uint64_t)(2 * M), (uint64_t)M, (uint64_t)a.batch};
    const uint64_t sa[2] = {(uint64_t)a.lda * 8, (uint64_t)a.strideA * 8};
    const uint32_t ba[3] = {32, 16, 1};
    if (encode_f32_map(&ma, a.A, 3, da, sa, ba, false)) return kTmaNotApplicable;
    const uint64_t db[3] = {(uint64_t)(2 * M), (uint64_t)a.n, (uint64_t)a.batch};
    const uint64_t sb[2] = {(uint64_t)a.ldb * 8, (uint64_t)a.strideB * 8};
    const uint32_t bb[3] = {32, (uint32_t)W, 1};
    if (encode_f32_map(&mb, a.B, 3, db, sb, bb, true)) return kTmaNotApplicable;
    auto kern = small_tma_c64_kernel<M, W, ST>;
    static_assert(U::kSmem <= 227 * 1024, "c64 TMA kernel shared memory");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)U::kSmem);
    if (e != cudaSuccess) return cuda_status(e);
    int *status = nullptr;
    const int rc = device_status_word(&status);
    if (rc) return rc;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 152;
    const int64_t items = a.batch * ((a.n + W - 1) / W);
    int64_t ctas = (items + U::kUnits - 1) / U::kUnits;
    if (ctas > sms) ctas = sms;  // persistent: one CTA per SM
    kern<<<(unsigned)ctas, U::kThreads, U::kSmem, st>>>(ma, mb, (int)a.n, alpha, items, status);
    return launch_status();
}

template <int M, int W>
static int launch_tma_c64_m(const SmallArgs &a, cudaStream_t st) {
    return launch_tma_c64_mw<M, W, 1>(a, st);
}

inline int launch_tma_c64(const SmallArgs &a, cudaStream_t st) {
    if (a.layout != 0 || a.n <= 16 || a.batch >= (int64_t(1) << 31) || a.n >= (int64_t(1) << 31))
        return kTmaNotApplicable;
    if (((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) != 0 || a.lda % 2 ||
        a.ldb % 2 || a.strideA % 2 || a.strideB % 2)
        return kTmaNotApplicable;
    const bool narrow = a.n <= 32;
    const int64_t items = a.batch * (narrow ? 1 : (a.n + 63) / 64);
    if (items < 2 * 152) return kTmaNotApplicable;  // a handful of items: the per-system kernels
    switch (a.m) {
        case 32: return narrow ? launch_tma_c64_m<32, 32>(a, st) : launch_tma_c64_m<32, 64>(a, st);
        case 48: return narrow ? launch_tma_c64_m<48, 32>(a, st) : launch_tma_c64_m<48, 64>(a, st);
        case 64: return narrow ? launch_tma_c64_m<64, 32>(a, st) : launch_tma_c64_m<64, 64>(a, st);
        default: return kTmaNotApplicable;
    }
}

}  // namespace trsm
