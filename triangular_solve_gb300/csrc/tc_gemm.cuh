// f32 products of the blocked solve on the fifth-generation tensor cores
// (tcgen05, sm_100 family):  C = beta*C + gamma * A X
// with A (M x K) and X (K x N) stored K-major: the trailing update (A the
// L panel or L_panel D_t^-1, X the block row), the block apply (A = D_t^-1,
// lower triangular) and the scaled panel (L_panel D_t^-1)^T (A = D_t^-T,
// upper triangular).
//
// f32 accuracy from TF32 tensor cores: each operand is split into a TF32
// head and a TF32 tail (a = hi + lo, hi = tf32(a), lo = tf32(a - hi)) by a
// preprocessing pass (or by the epilogue that produced it), and the product
// is accumulated in FP32 as
//     A_hi X_hi + A_hi X_lo + A_lo X_hi
// (the dropped A_lo X_lo term is ~2^-22 relative).
//
// Persistent kernel on CTA pairs (clusters of two, tcgen05 cta_group::2):
// each pair takes 256 x 256 output tiles in turn (of up to three independent
// products per launch); each CTA of the pair holds 128 rows of A and 128
// rows of X per K slab, and six warps:
//   warp 0  TMA producer: 2-D tensor loads of its four operand halves of a
//           16-deep K slab into a six-stage shared-memory ring (64-byte
//           swizzle), completion counted on the even CTA's "full" mbarrier;
//           the ring runs on from one tile to the next;
//   warp 1  (even CTA) MMA issuer: one elected thread issues the pair's
//           tcgen05.mma (kind::tf32, M = 256, N = 256, K = 8) into one of two
//           FP32 accumulators in tensor memory (2 x 256 columns in each CTA);
//           tcgen05.commit frees each stage and signals "accumulator full" in
//           both CTAs;
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes, release of the
//           accumulator to the even CTA, then the output straight to global
//           memory (coalesced per column) while the MMAs of the next tile run.
// Every mbarrier wait is bounded: when a wait expires the kernel records
// TRSM_ERR_DEVICE_TIMEOUT in a device status word and the CTA unwinds
// (no hang): it waits (bounded) for the loads and MMAs in flight, meets its
// peer at the cluster barrier, then releases its tensor memory.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "mbarrier.cuh"

namespace trsm {

// Tile shape: 128 rows of A and 256 columns per CTA accumulator, K slabs of
// 16 (64-byte K-major rows, 64-byte swizzle; measured on GB300: 32-deep
// slabs with the 128-byte swizzle were 1.5-10% slower).
constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 16;
static_assert(TC_BK == 16 || TC_BK == 32, "stage depth");
constexpr int kTileGroup = 8;  // row tiles per group of the tile order
constexpr uint32_t TC_ROW_BYTES = TC_BK * 4;  // a K-major tile row: the swizzle span
constexpr uint32_t TC_TMEM_COLS = 512;        // two 256-column FP32 accumulators

// out = beta*C + gamma*(A X) (beta_zero: out = gamma*(A X), C not read),
// stored to C; with xhi set, out is also stored split (TF32 head/tail) and
// K-major, xhi[col * ldxs + row], as the X operand of a later product, for
// the rows below xrows.
// a_lower: A is lower triangular, so a row tile stops its K loop at its last
// row (a_lower = 2: K interleaves real and imaginary parts, two K per row).
// cplx: the product is the real form of a complex one, output columns 2j
// and 2j+1 being the real and imaginary parts of complex column j of C
// (interleaved, ldc counted in floats); beta = beta + i*beta_im and
// gamma = gamma + i*gamma_im multiply complex values; with xhi set the
// split copy is the X' operand of tc_update_c64: row 2j = [Re | -Im],
// row 2j+1 = [Im | Re], halves ldxs/2 apart.
// a_upper: A is upper triangular, a row tile starts its K loop at its first
// row (a_upper = 2: interleaved K).  C == nullptr (with beta_zero and xhi
// set): only the split copy is stored.  xmode picks the layout of a complex
// split copy: 0 the X' rows above with [Re | Im] halves; 1 the same rows with
// interleaved K (row 2j = [Re x_0, -Im x_0, Re x_1, ...], row 2j+1 =
// [Im x_0, Re x_0, ...]); 2 the output transposed as the A' operand of a
// later product, interleaved: xhi[j * ldxs + 2 * row + {0, 1}] = {Re, Im}.
struct TcArgs {
    int64_t M, N, K;
    float *C;
    int64_t ldc;
    float beta, beta_im, gamma, gamma_im;
    int beta_zero, a_lower, a_upper, cplx, xmode;
    float *xhi, *xlo;
    int64_t ldxs, xrows;
};

// One launch computes up to kTcMaxProblems independent products: their tiles
// are numbered one problem after the other (problem i owns tiles
// tile_begin .. tile_begin + tiles_m * tiles_n - 1), and the persistent CTAs
// walk the concatenated list, so a small or triangular product fills the
// rounds of a larger one instead of running a partly idle launch of its own.
constexpr int kTcMaxProblems = 3;
struct TcProblem {
    CUtensorMap a_hi, a_lo, x_hi, x_lo;  // K-major operand tiles, head and tail
    TcArgs g;
    int tile_begin, tiles_m, tiles_n, nk;
};
struct TcLaunch {
    TcProblem p[kTcMaxProblems];
    int np, ntiles;
    int *status;  // device status word (0 = ok)
};

// Shared-memory matrix descriptor of a K-major tile with TC_ROW_BYTES-byte
// rows and the matching swizzle (128 B: mode 2, 64 B: mode 4); 8-row groups
// 8 * TC_ROW_BYTES apart.
__device__ __forceinline__ uint64_t tile_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);                  // start address
    d |= (uint64_t)1 << 16;                                   // leading byte offset (unused when swizzled)
    d |= (uint64_t)((8 * TC_ROW_BYTES) >> 4) << 32;           // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                                   // descriptor version for tcgen05
    d |= (uint64_t)(TC_ROW_BYTES == 128 ? 2 : 4) << 61;       // swizzle mode
    return d;
}

// Instruction descriptor: kind::tf32, FP32 accumulator, A and B K-major.
__host__ __device__ constexpr uint32_t tf32_idesc(int m, int n) {
    return (1u << 4)                     // D format F32
           | (2u << 7)                   // A format TF32
           | (2u << 10)                  // B format TF32
           | ((uint32_t)(n >> 3) << 17)  // N / 8
           | ((uint32_t)(m >> 4) << 24); // M / 16
}

// Round to TF32, nearest (ties away from zero).
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// ---------------------------------------------------------------------------
// The CTA pair (tcgen05 cta_group::2): the two CTAs of a cluster compute one
// 256 x 256 output tile.  Each holds 128 rows of A and 128 rows of X per
// K slab (32 KB a stage instead of 48: six stages in the same 192 KB), the
// pair's MMA (M = 256, N = 256, K = 8), issued by the even CTA, reads both
// CTAs' shared memory and leaves each CTA its 128 rows x 256 columns of the
// accumulator in its own tensor memory.
//   producer (both CTAs)  loads its halves; the loads complete on the even
//                         CTA's "full" barrier, which expects the pair's bytes;
//   MMA (even CTA)        commits "empty" and "accumulator full" to both CTAs;
//   epilogue (both CTAs)  drains its accumulator rows and arrives on the even
//                         CTA's "accumulator empty" (eight warps).
// Against one CTA per 128 x 256 tile, the operand feed per SM drops by a
// third and the tensor core's shared-memory reads per MMA from 12 KB to 8 KB
// (measured on GB300: f32 m = 16384 17.6 -> 16.0 ms, c64 60.3 -> 53.2 ms).
// ---------------------------------------------------------------------------
constexpr int TC2_STAGES = 6;
constexpr uint32_t TC2_A_BYTES = TC_BM * TC_BK * 4;        // 128 rows of A per CTA
constexpr uint32_t TC2_B_BYTES = (TC_BN / 2) * TC_BK * 4;  // 128 rows of X per CTA
constexpr uint32_t TC2_STAGE_BYTES = 2 * TC2_A_BYTES + 2 * TC2_B_BYTES;
constexpr uint32_t kTc2BarBytes = 256;
constexpr uint32_t kTc2TmemSlot = 8u * (2 * TC2_STAGES + 5);
static_assert(kTc2TmemSlot + 4 <= kTc2BarBytes, "barriers and TMEM slot fit their region");
constexpr size_t TC2_SMEM = 1024 + TC2_STAGES * TC2_STAGE_BYTES + kTc2BarBytes;
constexpr int TC2_PAIR_M = 2 * TC_BM;  // output rows of a pair tile

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr) : "memory");
}
// 2-D tile load into this CTA's shared memory, completing on a barrier of
// either CTA of the pair (cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the barrier at this offset in both CTAs of the pair once the
// pair's MMAs issued so far have completed
__device__ __forceinline__ void mma_commit_pair_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
            bar),
        "h"((uint16_t)3)
        : "memory");
}
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcLaunch P) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-byte alignment for the swizzled tiles
    unsigned char *sbase = smem_raw + (base - raw);
    const uint32_t bars = base + TC2_STAGES * TC2_STAGE_BYTES;
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (TC2_STAGES + s); };
    auto acc_full = [&](int a) { return bars + 8u * (2 * TC2_STAGES + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (2 * TC2_STAGES + 2 + a); };
    const uint32_t drain = bars + 8u * (2 * TC2_STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + TC2_STAGES * TC2_STAGE_BYTES + kTc2TmemSlot);
    __shared__ int abort_flag;
    __shared__ TcArgs s_args[kTcMaxProblems];
    __shared__ int4 s_tiles[kTcMaxProblems];  // tile_begin, tiles_m (pair rows), tiles_n, nk

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = (int)blockIdx.x >> 1, npairs = (int)gridDim.x >> 1;
    const int ntiles = P.ntiles, np = P.np;
    auto tile_of = [&](int t, int &pq, int &tm, int &tn) {
        pq = 0;
        while (pq + 1 < np && t >= s_tiles[pq + 1].x) ++pq;
        const int4 q = s_tiles[pq];
        const int u = t - q.x;
        const int per = kTileGroup * q.z;
        const int grp = u / per, rem = u - grp * per;
        const int gsize = min(kTileGroup, q.y - grp * kTileGroup);
        tm = grp * kTileGroup + rem % gsize;
        tn = rem / gsize;
    };
    auto k_range = [&](int pq, int m0, int &kb0, int &kb1) {
        const int nk = s_tiles[pq].w, lower = s_args[pq].a_lower;
        kb0 = s_args[pq].a_upper * m0 / TC_BK;
        kb1 = lower ? min(nk, lower * (m0 + TC2_PAIR_M) / TC_BK) : nk;
    };

    if (threadIdx.x < np) {
        const TcProblem &q = P.p[threadIdx.x];
        s_args[threadIdx.x] = q.g;
        s_tiles[threadIdx.x] = make_int4(q.tile_begin, q.tiles_m, q.tiles_n, q.nk);
    }
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < TC2_STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 8);  // four epilogue warps in each CTA
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(tmem_slot)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anything signals them
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    auto aborted = [&]() { return *(volatile int *)&abort_flag != 0; };
    auto fail = [&]() {
        record_timeout(P.status);
        abort_flag = 1;
    };

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int t = pair; t < ntiles && !aborted(); t += npairs) {
                int pq, tm, tn;
                tile_of(t, pq, tm, tn);
                const TcProblem &q = P.p[pq];
                const int m0 = tm * TC2_PAIR_M, n0 = tn * TC_BN;
                const int ya = m0 + TC_BM * (int)rank, yx = n0 + (TC_BN / 2) * (int)rank;
                int kb0, kb1;
                k_range(pq, m0, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % TC2_STAGES;
                    if (it >= TC2_STAGES && !mbar_wait(empty(s), ((it / TC2_STAGES) - 1) & 1)) {
                        fail();
                        break;
                    }
                    if (leader) mbar_expect_tx(full(s), 2 * TC2_STAGE_BYTES);
                    const uint32_t st = base + s * TC2_STAGE_BYTES, fb = map_to_rank(full(s), 0);
                    const int kx = kb * TC_BK;
                    tma_load_2d_pair(st, &q.a_hi, kx, ya, fb);
                    tma_load_2d_pair(st + TC2_A_BYTES, &q.a_lo, kx, ya, fb);
                    tma_load_2d_pair(st + 2 * TC2_A_BYTES, &q.x_hi, kx, yx, fb);
                    tma_load_2d_pair(st + 2 * TC2_A_BYTES + TC2_B_BYTES, &q.x_lo, kx, yx, fb);
                }
            }
            if (aborted() && leader) {
                // the pair's loads counted on these barriers land before shared memory goes away
                for (int j = (it > TC2_STAGES ? it - TC2_STAGES : 0); j < it; ++j)
                    if (!mbar_wait(full(j % TC2_STAGES), (j / TC2_STAGES) & 1)) record_timeout(P.status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = tf32_idesc(TC2_PAIR_M, TC_BN);
            int it = 0, i = 0;
            for (int t = pair; t < ntiles && !aborted(); t += npairs, ++i) {
                const int a = i & 1;
                if (i >= 2 && !mbar_wait(acc_empty(a), ((i >> 1) - 1) & 1)) {
                    fail();
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(a * TC_BN);
                int pq, tm, tn;
                tile_of(t, pq, tm, tn);
                int kb0, kb1;
                k_range(pq, tm * TC2_PAIR_M, kb0, kb1);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % TC2_STAGES;
                    if (!mbar_wait(full(s), (it / TC2_STAGES) & 1)) {
                        fail();
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
                    const uint32_t st = base + s * TC2_STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 8; ++kk) {
                        const uint64_t a_hi = tile_desc(st + kk * 32);
                        const uint64_t a_lo = tile_desc(st + TC2_A_BYTES + kk * 32);
                        const uint64_t x_hi = tile_desc(st + 2 * TC2_A_BYTES + kk * 32);
                        const uint64_t x_lo = tile_desc(st + 2 * TC2_A_BYTES + TC2_B_BYTES + kk * 32);
                        mma_tf32_pair(d, a_hi, x_hi, idesc, kb != kb0 || kk != 0);
                        mma_tf32_pair(d, a_hi, x_lo, idesc, 1);
                        mma_tf32_pair(d, a_lo, x_hi, idesc, 1);
                    }
                    mma_commit_pair_both(empty(s));  // both CTAs' stage s is free once these MMAs have read it
                }
                mma_commit_pair_both(acc_full(a));  // accumulator a complete (or abandoned) in both CTAs
                if (!ok) break;
            }
            mma_commit_pair_local(drain);
            if (!mbar_wait(drain, 0)) record_timeout(P.status);
        }
    } else {
        // epilogue warps 2..5: TMEM lanes 32*(warp % 4) .. +31 of this CTA's
        // 128 accumulator rows
        const int quarter = warp & 3;
        int i = 0;
        for (int t = pair; t < ntiles; t += npairs, ++i) {
            const int a = i & 1;
            int pq, tm, tn;
            tile_of(t, pq, tm, tn);
            const TcArgs &g = s_args[pq];
            const int m0 = tm * TC2_PAIR_M + TC_BM * (int)rank, n0 = tn * TC_BN;
            const int64_t gr = m0 + 32 * quarter + lane;
            const bool row_ok = gr < g.M;
            // loop invariants of the tile, hoisted: the column loops below
            // are unrolled, and a full column tile storing only C (the
            // update) runs without per-element checks
            float *const C = g.C;
            const int64_t ldc = g.ldc, N = g.N;
            const float beta = g.beta, gamma = g.gamma;
            const bool cplx = g.cplx != 0, load_c = !g.beta_zero && row_ok;
            const bool real_full = !cplx && n0 + TC_BN <= N;  // a full column tile of a real product
            float *const xhi = g.xhi, *const xlo = g.xlo;
            const int64_t ldxs = g.ldxs;
            const bool emit = xhi != nullptr && gr < g.xrows;  // this row also goes out split
            const int xmode = g.xmode;
            float cnext[32];
            // element (gr, gc) of C
            auto coff = [&](int64_t gc) -> int64_t {
                return cplx ? (gc >> 1) * ldc + 2 * gr + (gc & 1) : gc * ldc + gr;
            };
            auto fetch = [&](int chunk, float(&dst)[32]) {
                const int64_t gc0 = n0 + chunk * 32;
                if (!load_c) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[j] = 0.f;
                } else if (real_full) {
                    const float *cp = C + gc0 * ldc + gr;
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[j] = cp[j * ldc];
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[j] = (gc0 + j < N) ? C[coff(gc0 + j)] : 0.f;
                }
            };
            fetch(0, cnext);
            if (!mbar_wait(acc_full(a), (i >> 1) & 1)) {
                if (lane == 0) fail();
                break;
            }
            if (aborted()) break;
            asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(a * TC_BN);
#pragma unroll 1
            for (int chunk = 0; chunk < TC_BN / 32; ++chunk) {
                float ccur[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) ccur[j] = cnext[j];
                if (chunk + 1 < TC_BN / 32) fetch(chunk + 1, cnext);
                uint32_t v[32];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                    "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                    "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                      "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
                      "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
                      "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(lane_addr + (uint32_t)(chunk * 32)));
                asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
                if (chunk + 1 == TC_BN / 32) {
                    // every TMEM read of accumulator a is done: hand it back
                    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_to_rank(acc_empty(a), 0));
                }
                if (row_ok && cplx) {
                    const float beta_im = g.beta_im, gamma_im = g.gamma_im;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int64_t gc = n0 + chunk * 32 + j;  // even: a (re, im) pair
                        if (gc < N) {
                            const float cr = ccur[j], ci = ccur[j + 1];
                            const float pr = __uint_as_float(v[j]), pi = __uint_as_float(v[j + 1]);
                            const float ar = fmaf(gamma, pr, -gamma_im * pi);
                            const float ai = fmaf(gamma, pi, gamma_im * pr);
                            const float orr = fmaf(beta, cr, fmaf(-beta_im, ci, ar));
                            const float oi = fmaf(beta, ci, fmaf(beta_im, cr, ai));
                            if (C) *reinterpret_cast<float2 *>(C + coff(gc)) = make_float2(orr, oi);
                            if (emit) {
                                auto put2 = [&](int64_t o, float x, float y) {  // a pair, 8-byte aligned
                                    const float hx = to_tf32(x), hy = to_tf32(y);
                                    *reinterpret_cast<float2 *>(xhi + o) = make_float2(hx, hy);
                                    *reinterpret_cast<float2 *>(xlo + o) = make_float2(to_tf32(x - hx), to_tf32(y - hy));
                                };
                                if (xmode == 2) {
                                    put2((gc >> 1) * ldxs + 2 * gr, orr, oi);
                                } else if (xmode == 1) {
                                    const int64_t re_row = gc * ldxs, im_row = re_row + ldxs;
                                    put2(re_row + 2 * gr, orr, -oi);
                                    put2(im_row + 2 * gr, oi, orr);
                                } else {
                                    const int64_t re_row = gc * ldxs, im_row = re_row + ldxs, half = ldxs / 2;
                                    auto put = [&](int64_t o, float x) {
                                        const float h = to_tf32(x);
                                        xhi[o] = h;
                                        xlo[o] = to_tf32(x - h);
                                    };
                                    put(re_row + gr, orr);
                                    put(re_row + half + gr, -oi);
                                    put(im_row + gr, oi);
                                    put(im_row + half + gr, orr);
                                }
                            }
                        }
                    }
                } else if (row_ok && real_full && C && !emit) {
                    float *cp = C + (n0 + chunk * 32) * ldc + gr;
#pragma unroll
                    for (int j = 0; j < 32; ++j) cp[j * ldc] = fmaf(beta, ccur[j], gamma * __uint_as_float(v[j]));
                } else if (row_ok && real_full && C) {
                    const int64_t gc0 = n0 + chunk * 32;
                    float *cp = C + gc0 * ldc + gr, *hp = xhi + gc0 * ldxs + gr, *lp = xlo + gc0 * ldxs + gr;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float o = fmaf(beta, ccur[j], gamma * __uint_as_float(v[j]));
                        const float h = to_tf32(o);
                        cp[j * ldc] = o;
                        hp[j * ldxs] = h;
                        lp[j * ldxs] = to_tf32(o - h);
                    }
                } else if (row_ok) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int64_t gc = n0 + chunk * 32 + j;
                        if (gc < N) {
                            const float o = fmaf(beta, ccur[j], gamma * __uint_as_float(v[j]));
                            if (C) C[gc * ldc + gr] = o;
                            if (emit) {
                                const float h = to_tf32(o);
                                xhi[gc * ldxs + gr] = h;
                                xlo[gc * ldxs + gr] = to_tf32(o - h);
                            }
                        }
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    cluster_sync();  // the pair's MMAs and loads are done with both CTAs' memory
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TC_TMEM_COLS)
                     : "memory");
    }
}

// a = hi + lo with hi, lo both TF32 (round to nearest): dst rows r, K-major,
//   hi[r * ldd + k] = tf32(src[r + k * ks]),  lo = tf32(src - hi)
// for r < R, k < Kc.  32 x 32 tiles through shared memory (src is read
// along r, dst written along k).

__global__ void split_tf32_kernel(const float *__restrict__ src, int64_t ks, int64_t R, int64_t Kc,
                                  float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    __shared__ float tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.x * 32, k0 = (int64_t)blockIdx.y * 32;
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + threadIdx.x, k = k0 + q;
        tile[q][threadIdx.x] = (r < R && k < Kc) ? src[r + k * ks] : 0.f;
    }
    __syncthreads();
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + q, k = k0 + threadIdx.x;
        if (r < R && k < Kc) {
            const float a = tile[threadIdx.x][q];
            const float h = to_tf32(a);
            hi[r * ldd + k] = h;
            lo[r * ldd + k] = to_tf32(a - h);
        }
    }
}

// The same split for a source that is K-major already:
//   hi[r * ldd + k] = tf32(src[r * ks + k]),  lo = tf32(src - hi).
__global__ void split_rows_tf32_kernel(const float *__restrict__ src, int64_t ks, int64_t R, int64_t Kc,
                                       float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= Kc) return;
    for (int64_t r = blockIdx.y; r < R; r += gridDim.y) {
        const float a = src[r * ks + k];
        const float h = to_tf32(a);
        hi[r * ldd + k] = h;
        lo[r * ldd + k] = to_tf32(a - h);
    }
}

// The same with 16-byte accesses (source rows, destination rows and Kc all
// multiples of four floats, both bases 16-byte aligned): four elements per
// thread, so the split streams at HBM speed.
__global__ void split_rows_tf32_v4_kernel(const float4 *__restrict__ src, int64_t ks4, int64_t R, int64_t Kc4,
                                          float4 *__restrict__ hi, float4 *__restrict__ lo, int64_t ldd4) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= Kc4) return;
    for (int64_t r = blockIdx.y; r < R; r += gridDim.y) {
        const float4 a = src[r * ks4 + k];
        const float4 h = make_float4(to_tf32(a.x), to_tf32(a.y), to_tf32(a.z), to_tf32(a.w));
        hi[r * ldd4 + k] = h;
        lo[r * ldd4 + k] = make_float4(to_tf32(a.x - h.x), to_tf32(a.y - h.y), to_tf32(a.z - h.z), to_tf32(a.w - h.w));
    }
}

// Operands of a complex (c64) product in real form, TF32 head/tail, K-major
// with K' = 2 Kc:
//   A' row r = [Re A(r, 0..Kc) | Im A(r, 0..Kc)]          (A column-major, ks)
//   X' row 2j = [Re X(.., j) | -Im X(.., j)],  row 2j+1 = [Im X(.., j) | Re X(.., j)]
//                                                          (X row-major, ks)
// so that A' X'^T gives Re(A X) in column 2j and Im(A X) in column 2j+1.
__global__ void split_c64_a_kernel(const float2 *__restrict__ src, int64_t ks, int64_t R, int64_t Kc,
                                   float *__restrict__ hi, float *__restrict__ lo) {
    __shared__ float2 tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.x * 32, k0 = (int64_t)blockIdx.y * 32;
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + threadIdx.x, k = k0 + q;
        tile[q][threadIdx.x] = (r < R && k < Kc) ? src[r + k * ks] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + q, k = k0 + threadIdx.x;
        if (r < R && k < Kc) {
            const float2 a = tile[threadIdx.x][q];
            const int64_t o = r * 2 * Kc + k;
            float h = to_tf32(a.x);
            hi[o] = h;
            lo[o] = to_tf32(a.x - h);
            h = to_tf32(a.y);
            hi[o + Kc] = h;
            lo[o + Kc] = to_tf32(a.y - h);
        }
    }
}

__global__ void split_c64_x_kernel(const float2 *__restrict__ src, int64_t ks, int64_t Kc, int64_t N,
                                   float *__restrict__ hi, float *__restrict__ lo) {
    __shared__ float2 tile[32][33];
    const int64_t j0 = (int64_t)blockIdx.x * 32, k0 = (int64_t)blockIdx.y * 32;
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t j = j0 + threadIdx.x, k = k0 + q;
        tile[q][threadIdx.x] = (j < N && k < Kc) ? src[k * ks + j] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    auto put = [&](int64_t o, float x) {
        const float h = to_tf32(x);
        hi[o] = h;
        lo[o] = to_tf32(x - h);
    };
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t j = j0 + q, k = k0 + threadIdx.x;
        if (j < N && k < Kc) {
            const float2 x = tile[threadIdx.x][q];
            const int64_t re = 2 * j * 2 * Kc, im = re + 2 * Kc;
            put(re + k, x.x);
            put(re + Kc + k, -x.y);
            put(im + k, x.y);
            put(im + Kc + k, x.x);
        }
    }
}

// Operands of the complex block apply in real form with interleaved K'
// (k' = 2k for the real part, 2k + 1 for the imaginary part), which keeps a
// lower-triangular A's K range a prefix:
//   A' row r = [Re A(r,0), Im A(r,0), Re A(r,1), ...]   (A column-major, ks)
//   X' row 2j = [Re X(0,j), -Im X(0,j), ...], row 2j+1 = [Im X(0,j), Re X(0,j), ...]
//                                                      (X column-major, ks)
__global__ void split_c64_ai_kernel(const float2 *__restrict__ src, int64_t ks, int64_t R, int64_t Kc,
                                    float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    __shared__ float2 tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.x * 32, k0 = (int64_t)blockIdx.y * 32;
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + threadIdx.x, k = k0 + q;
        tile[q][threadIdx.x] = (r < R && k < Kc) ? src[r + k * ks] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t r = r0 + q, k = k0 + threadIdx.x;
        if (r < R && k < Kc) {
            const float2 a = tile[threadIdx.x][q];
            const float hr = to_tf32(a.x), hi_ = to_tf32(a.y);
            const int64_t o = r * ldd + 2 * k;
            *reinterpret_cast<float2 *>(hi + o) = make_float2(hr, hi_);
            *reinterpret_cast<float2 *>(lo + o) = make_float2(to_tf32(a.x - hr), to_tf32(a.y - hi_));
        }
    }
}

__global__ void split_c64_xi_kernel(const float2 *__restrict__ src, int64_t ks, int64_t Kc, int64_t N,
                                    float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= Kc) return;
    for (int64_t j = blockIdx.y; j < N; j += gridDim.y) {
        const float2 x = src[j * ks + k];
        const float hr = to_tf32(x.x), hm = to_tf32(x.y);
        const float lr = to_tf32(x.x - hr), lm = to_tf32(x.y - hm);
        const int64_t re = 2 * j * ldd + 2 * k, im = re + ldd;
        *reinterpret_cast<float2 *>(hi + re) = make_float2(hr, -hm);
        *reinterpret_cast<float2 *>(lo + re) = make_float2(lr, -lm);
        *reinterpret_cast<float2 *>(hi + im) = make_float2(hm, hr);
        *reinterpret_cast<float2 *>(lo + im) = make_float2(lm, lr);
    }
}

// X' rows with interleaved K of the transpose of a column-major panel:
// X(k, i) = src[i + k * ks] (i < R, k < Kc), so row 2i of the output is
// [Re src(i, 0), -Im src(i, 0), Re src(i, 1), ...] and row 2i + 1 is
// [Im src(i, 0), Re src(i, 0), ...] (row stride ldd floats).  32 x 32 tiles
// through shared memory (src is read along i, the output written along k).
__global__ void split_c64_xt_kernel(const float2 *__restrict__ src, int64_t ks, int64_t R, int64_t Kc,
                                    float *__restrict__ hi, float *__restrict__ lo, int64_t ldd) {
    __shared__ float2 tile[32][33];
    const int64_t i0 = (int64_t)blockIdx.x * 32, k0 = (int64_t)blockIdx.y * 32;
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t i = i0 + threadIdx.x, k = k0 + q;
        tile[q][threadIdx.x] = (i < R && k < Kc) ? src[i + k * ks] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    for (int q = threadIdx.y; q < 32; q += blockDim.y) {
        const int64_t i = i0 + q, k = k0 + threadIdx.x;
        if (i < R && k < Kc) {
            const float2 x = tile[threadIdx.x][q];
            const float hr = to_tf32(x.x), hm = to_tf32(x.y);
            const float lr = to_tf32(x.x - hr), lm = to_tf32(x.y - hm);
            const int64_t re = 2 * i * ldd + 2 * k, im = re + ldd;
            *reinterpret_cast<float2 *>(hi + re) = make_float2(hr, -hm);
            *reinterpret_cast<float2 *>(lo + re) = make_float2(lr, -lm);
            *reinterpret_cast<float2 *>(hi + im) = make_float2(hm, hr);
            *reinterpret_cast<float2 *>(lo + im) = make_float2(lm, lr);
        }
    }
}

}  // namespace trsm
