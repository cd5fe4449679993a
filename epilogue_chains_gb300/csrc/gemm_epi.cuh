// gemm_epi.cuh -- the epilogue stages of the GEMM chain (+bias, GELU(erf), +residual) and fp16
// packing, shared by the tile GEMM (gemm.cu) and the decode GEMM (gemm_decode.cu).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace fc {
namespace {

// ------------------------------------------------------------------------------ epilogue math
// Stages of the chain after the GEMM: 1 = +bias, 2 = GELU(erf), 3 = +residual.
//
// GELU(v) = v/2 (1 + erf(v/sqrt2)).  1 + erf(x) is evaluated as erfc(-x) for x < 0 and as
// 2 - erfc(x) for x >= 0, so there is no cancellation for strongly negative v (where 1 + erf(x)
// is tiny).  erfc(z), z >= 0, is the Chebyshev-fitted approximation "erfcc" of Press, Teukolsky,
// Vetterling & Flannery, Numerical Recipes (2nd ed., §6.2): erfc(z) = t exp(-z^2 + P(t)),
// t = 1/(1 + z/2), fractional error below 1.2e-7 for every z >= 0 -- far below the fp16 output
// resolution.  Cost per element: one reciprocal and one ex2 (MUFU), the rest in packed fp32x2
// instructions (sm_100+), which evaluate two elements per instruction.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// GELU of two values at once
__device__ __forceinline__ float2 gelu_erf2(float2 v) {
    const float2 z = __fmul2_rn(make_float2(fabsf(v.x), fabsf(v.y)), f2(0.70710678118654752f));
    const float2 d = __ffma2_rn(f2(0.5f), z, f2(1.0f));
    const float2 t = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    float2 p = f2(0.17087277f);
    p = __ffma2_rn(p, t, f2(-0.82215223f));
    p = __ffma2_rn(p, t, f2(1.48851587f));
    p = __ffma2_rn(p, t, f2(-1.13520398f));
    p = __ffma2_rn(p, t, f2(0.27886807f));
    p = __ffma2_rn(p, t, f2(-0.18628806f));
    p = __ffma2_rn(p, t, f2(0.09678418f));
    p = __ffma2_rn(p, t, f2(0.37409196f));
    p = __ffma2_rn(p, t, f2(1.00002368f));
    p = __ffma2_rn(p, t, f2(-1.26551223f));
    const float2 a = __fmul2_rn(__ffma2_rn(make_float2(-z.x, -z.y), z, p), f2(1.44269504088896341f));
    const float2 e = __fmul2_rn(t, make_float2(ex2_approx(a.x), ex2_approx(a.y)));
    const float2 s = make_float2(v.x >= 0.0f ? 2.0f - e.x : e.x, v.y >= 0.0f ? 2.0f - e.y : e.y);
    return __fmul2_rn(__fmul2_rn(f2(0.5f), v), s);
}
__device__ __forceinline__ float gelu_erf(float v) { return gelu_erf2(make_float2(v, v)).x; }

// apply stages first..last (inclusive, 1..3) to v
__device__ __forceinline__ float apply_stages(float v, int first, int last, float b, float r) {
    if (first <= 1 && last >= 1) v += b;
    if (first <= 2 && last >= 2) v = gelu_erf(v);
    if (first <= 3 && last >= 3) v += r;
    return v;
}
// the same on two values
__device__ __forceinline__ float2 apply_stages2(float2 v, int first, int last, float2 b, float2 r) {
    if (first <= 1 && last >= 1) v = __fadd2_rn(v, b);
    if (first <= 2 && last >= 2) v = gelu_erf2(v);
    if (first <= 3 && last >= 3) v = __fadd2_rn(v, r);
    return v;
}

// the same with the last stage fixed at compile time (stages 1..LAST), so that a loop over many
// values is one branch-free block whose independent GELU chains the compiler can interleave
template <int LAST>
__device__ __forceinline__ float2 apply_stages2_upto(float2 v, float2 b, float2 r) {
    if constexpr (LAST >= 1) v = __fadd2_rn(v, b);
    if constexpr (LAST >= 2) v = gelu_erf2(v);
    if constexpr (LAST >= 3) v = __fadd2_rn(v, r);
    return v;
}
template <int N>
struct IntC {
    static constexpr int value = N;
};

__device__ __forceinline__ void unpack_h8(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 pack_h8(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace
}  // namespace fc
