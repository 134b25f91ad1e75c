// Shared device helpers of the GB300 TRSM library: element types and their
// arithmetic, asynchronous global->shared copies, launch checking.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/trsm.h"

namespace trsm {

// ----------------------------------------------------------------------------
// Element types.  Complex values are interleaved {re, im} (float2 / double2),
// the layout of torch.complex64 / complex128.
// ----------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float>   { using Real = float;  static constexpr bool kComplex = false; };
template <> struct Elem<double>  { using Real = double; static constexpr bool kComplex = false; };
template <> struct Elem<float2>  { using Real = float;  static constexpr bool kComplex = true; };
template <> struct Elem<double2> { using Real = double; static constexpr bool kComplex = true; };

template <typename T> __host__ __device__ __forceinline__ T zero_of();
template <> __host__ __device__ __forceinline__ float zero_of<float>() { return 0.f; }
template <> __host__ __device__ __forceinline__ double zero_of<double>() { return 0.0; }
template <> __host__ __device__ __forceinline__ float2 zero_of<float2>() { return make_float2(0.f, 0.f); }
template <> __host__ __device__ __forceinline__ double2 zero_of<double2>() { return make_double2(0.0, 0.0); }
template <typename T> __device__ __forceinline__ T one_of();
template <> __device__ __forceinline__ float one_of<float>() { return 1.f; }
template <> __device__ __forceinline__ double one_of<double>() { return 1.0; }
template <> __device__ __forceinline__ float2 one_of<float2>() { return make_float2(1.f, 0.f); }
template <> __device__ __forceinline__ double2 one_of<double2>() { return make_double2(1.0, 0.0); }

// a * b
__device__ __forceinline__ float mul(float a, float b) { return a * b; }
__device__ __forceinline__ double mul(double a, double b) { return a * b; }
__device__ __forceinline__ float2 mul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
__device__ __forceinline__ double2 mul(double2 a, double2 b) {
    return make_double2(fma(a.x, b.x, -a.y * b.y), fma(a.x, b.y, a.y * b.x));
}

// c - a * b (the substitution update), fused where the pipe allows.
__device__ __forceinline__ float fms(float a, float b, float c) { return fmaf(-a, b, c); }
__device__ __forceinline__ double fms(double a, double b, double c) { return fma(-a, b, c); }
__device__ __forceinline__ float2 fms(float2 a, float2 b, float2 c) {
    float re = fmaf(-a.x, b.x, c.x);
    float im = fmaf(-a.x, b.y, c.y);
    re = fmaf(a.y, b.y, re);
    im = fmaf(-a.y, b.x, im);
    return make_float2(re, im);
}
__device__ __forceinline__ double2 fms(double2 a, double2 b, double2 c) {
    double re = fma(-a.x, b.x, c.x);
    double im = fma(-a.x, b.y, c.y);
    re = fma(a.y, b.y, re);
    im = fma(-a.y, b.x, im);
    return make_double2(re, im);
}

// c + a * b
__device__ __forceinline__ float fma_(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fma_(double a, double b, double c) { return fma(a, b, c); }
__device__ __forceinline__ float2 fma_(float2 a, float2 b, float2 c) {
    float re = fmaf(a.x, b.x, c.x);
    float im = fmaf(a.x, b.y, c.y);
    re = fmaf(-a.y, b.y, re);
    im = fmaf(a.y, b.x, im);
    return make_float2(re, im);
}
__device__ __forceinline__ double2 fma_(double2 a, double2 b, double2 c) {
    double re = fma(a.x, b.x, c.x);
    double im = fma(a.x, b.y, c.y);
    re = fma(-a.y, b.y, re);
    im = fma(a.y, b.x, im);
    return make_double2(re, im);
}

// a - b
__device__ __forceinline__ float sub_(float a, float b) { return a - b; }
__device__ __forceinline__ double sub_(double a, double b) { return a - b; }
__device__ __forceinline__ float2 sub_(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ double2 sub_(double2 a, double2 b) { return make_double2(a.x - b.x, a.y - b.y); }

// 1 / d.  Real: the IEEE division operator.  Complex: Smith's 1962 method
// (R. L. Smith, "Algorithm 116: Complex division", CACM 5(8)), which scales
// by the larger of |re|, |im| so that the squared modulus is never formed.
__device__ __forceinline__ float recip(float d) { return 1.0f / d; }
__device__ __forceinline__ double recip(double d) { return 1.0 / d; }
template <typename C, typename R>
__device__ __forceinline__ C recip_smith(R c, R d) {
    C r;
    if (fabs(c) >= fabs(d)) {
        R q = d / c;
        R den = c + d * q;
        r.x = R(1) / den;
        r.y = -q / den;
    } else {
        R q = c / d;
        R den = c * q + d;
        r.x = q / den;
        r.y = R(-1) / den;
    }
    return r;
}
__device__ __forceinline__ float2 recip(float2 d) { return recip_smith<float2, float>(d.x, d.y); }
__device__ __forceinline__ double2 recip(double2 d) { return recip_smith<double2, double>(d.x, d.y); }

// v == 1 exactly
__device__ __forceinline__ bool is_one(float v) { return v == 1.f; }
__device__ __forceinline__ bool is_one(double v) { return v == 1.0; }
__device__ __forceinline__ bool is_one(float2 v) { return v.x == 1.f && v.y == 0.f; }
__device__ __forceinline__ bool is_one(double2 v) { return v.x == 1.0 && v.y == 0.0; }

template <typename T> __device__ __forceinline__ T ldg(const T *p) { return __ldg(p); }

// ----------------------------------------------------------------------------
// Paired FP32 arithmetic (fma.rn.f32x2, sm_100 and later): two independent
// single-precision FMAs in one instruction, operands packed in 64 bits
// (low half = first element).  Halves the issue slots of FP32 FMA work.
// ----------------------------------------------------------------------------
using f32x2 = unsigned long long;
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// a * b + c, element-wise on both halves
__device__ __forceinline__ f32x2 ffma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// ----------------------------------------------------------------------------
// cp.async (LDGSTS): global -> shared copies that bypass registers.  Sizes
// 4, 8 and 16 bytes; both addresses must be aligned to the size.
// ----------------------------------------------------------------------------
template <int BYTES>
__device__ __forceinline__ void cp_async(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    if constexpr (BYTES == 16) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
    } else if constexpr (BYTES == 8) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
    } else {
        static_assert(BYTES == 4, "cp.async size");
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ----------------------------------------------------------------------------
// Host-side status helpers.
// ----------------------------------------------------------------------------
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? TRSM_SUCCESS : TRSM_ERR_CUDA_BASE + (int)e; }
inline int launch_status() { return cuda_status(cudaGetLastError()); }

}  // namespace trsm
