// swiglu.cuh -- h = bf16(silu(g) u) for packed bf16 pairs: the SwiGLU
// evaluation shared by the fused SwiGLU + quantize kernel and the grouped GEMM's
// SwiGLU epilogue, so that both give the same bits for the same g and u.
#pragma once

#include "common.cuh"

namespace nvfp4 {

// silu(g) u for the two bf16 values of a word pair, in binary32 with packed
// (FP32x2) arithmetic: e = exp(-|g|) = 2^(-|g| log2 e) lies in (0, 1] and never
// overflows; sigma(g) = 1/(1+e) for g >= 0 and e/(1+e) for g < 0 (the two forms
// of the logistic function); h = bf16((g sigma(g)) u).  ex2.approx and
// rcp.approx are each within a few binary32 ulps and the rounding of the
// exponent argument adds at most ~2^-17 relative for |g| up to 150, far inside
// half a bf16 ulp (2^-9), so h is within one bf16 ulp of bf16(silu(g) u)
// evaluated exactly while e stays a normal float or a subnormal with ten or
// more significant bits (g >= -96; below that |silu(g)| < 1e-39).
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t swiglu_pair(uint32_t g2, uint32_t u2) {
    const float2 g = make_float2(bf16lo(g2), bf16hi(g2));
    const uint32_t a2 = g2 & 0x7FFF7FFFu;
    const float2 t = __fmul2_rn(make_float2(bf16lo(a2), bf16hi(a2)), make_float2(-kLog2e, -kLog2e));
    const float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    const float2 d = __fadd2_rn(e, make_float2(1.0f, 1.0f));
    const float2 num = make_float2(g.x < 0.0f ? e.x : 1.0f, g.y < 0.0f ? e.y : 1.0f);
    const float2 sig = __fmul2_rn(num, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
    const float2 h = __fmul2_rn(__fmul2_rn(g, sig), make_float2(bf16lo(u2), bf16hi(u2)));
    const __nv_bfloat162 hb = __floats2bfloat162_rn(h.x, h.y);
    return *reinterpret_cast<const uint32_t*>(&hb);
}

}  // namespace nvfp4
