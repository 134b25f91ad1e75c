// Throughput probe for the arithmetic pipes the solver's kernels run on:
// FP32 FFMA, FP64 DFMA and the FP64 warp-level MMA (mma.sync m8n8k4 f64).
// Every thread runs independent FMA chains so that issue, not latency,
// limits the rate.  The result is the denominator of the "alu" roofline of
// the FP64-bound kernels and the FFMA reference of the FP32 ones.
//
// Built into its own library (libtrsm_peaks.so), separate from the solver.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kChains = 8;

__global__ void ffma_loop(float *out, float a, float b, int iters) {
    float acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = threadIdx.x * 1e-3f + c;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) acc[c] = fmaf(acc[c], a, b);
    }
    float s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c];
    if (s == 12345.678f) out[threadIdx.x] = s;  // keeps the loop live
}

__global__ void dfma_loop(double *out, double a, double b, int iters) {
    double acc[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc[c] = threadIdx.x * 1e-3 + c;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) acc[c] = fma(acc[c], a, b);
    }
    double s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += acc[c];
    if (s == 12345.678) out[threadIdx.x] = s;
}

// Paired FP32 FMA (fma.rn.f32x2): two FMAs per instruction.
__global__ void ffma2_loop(float *out, float a, float b, int iters) {
    unsigned long long acc[kChains];
    unsigned long long av, bv;
    asm("mov.b64 %0, {%1, %2};" : "=l"(av) : "f"(a), "f"(a));
    asm("mov.b64 %0, {%1, %2};" : "=l"(bv) : "f"(b), "f"(b));
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        const float lo = threadIdx.x * 1e-3f + c, hi = lo + 0.5f;
        asm("mov.b64 %0, {%1, %2};" : "=l"(acc[c]) : "f"(lo), "f"(hi));
    }
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[c]) : "l"(av), "l"(bv));
    }
    float s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[c]));
        s += lo + hi;
    }
    if (s == 12345.678f) out[threadIdx.x] = s;
}

// D(8x8) += A(8x4) B(4x8), f64; 4 independent accumulators per warp.
__global__ void dmma_loop(double *out, double a, double b, int iters) {
    double d[4][2];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c][0] = d[c][1] = threadIdx.x * 1e-3 + c;
    const double av = a + threadIdx.x * 1e-9, bv = b - threadIdx.x * 1e-9;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            asm volatile(
                "mma.sync.aligned.m8n8k4.row.col.f64.f64.f64.f64 {%0,%1}, {%2}, {%3}, {%0,%1};\n"
                : "+d"(d[c][0]), "+d"(d[c][1])
                : "d"(av), "d"(bv));
        }
    }
    double s = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) s += d[c][0] + d[c][1];
    if (s == 12345.678) out[threadIdx.x] = s;
}

}  // namespace

extern "C" {

// kind 0: FFMA, 1: DFMA, 2: DMMA (m8n8k4), 3: FFMA2 (fma.rn.f32x2).  Returns TFLOP/s (2 flops per
// multiply-add) measured with CUDA events over `reps` launches, or a
// negative value on a CUDA error.
double trsm_probe_pipe_tflops(int kind, int reps) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    void *buf = nullptr;
    if (cudaMalloc(&buf, 4096 * sizeof(double)) != cudaSuccess) return -2;
    const int threads = 256, blocks = sms * 8;
    const int iters = kind == 0 ? 16384 : (kind == 1 ? 512 : (kind == 2 ? 256 : 8192));
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    auto launch = [&]() {
        if (kind == 0) ffma_loop<<<blocks, threads>>>((float *)buf, 0.999f, 1e-3f, iters);
        else if (kind == 3) ffma2_loop<<<blocks, threads>>>((float *)buf, 0.999f, 1e-3f, iters);
        else if (kind == 1) dfma_loop<<<blocks, threads>>>((double *)buf, 0.999, 1e-3, iters);
        else dmma_loop<<<blocks, threads>>>((double *)buf, 0.999, 1e-3, iters);
    };
    launch();  // warm-up
    cudaEventRecord(e0);
    for (int r = 0; r < reps; ++r) launch();
    cudaEventRecord(e1);
    cudaError_t err = cudaEventSynchronize(e1);
    float ms = 0;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(buf);
    if (err != cudaSuccess || cudaGetLastError() != cudaSuccess) return -3;
    double fmas;
    if (kind == 2) fmas = (double)blocks * (threads / 32) * 4 * iters * (8.0 * 8 * 4);
    else if (kind == 3) fmas = 2.0 * blocks * threads * kChains * iters;
    else fmas = (double)blocks * threads * kChains * iters;
    return 2.0 * fmas * reps / (ms * 1e-3) / 1e12;
}

}  // extern "C"
