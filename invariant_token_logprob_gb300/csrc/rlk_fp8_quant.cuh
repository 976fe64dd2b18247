// rlk_fp8_quant.cuh -- the per-element arithmetic of the e4m3 quantisation
// (row scale amax / 448, the division by it, the RNE conversion), shared by
// the quantiser kernels and by the LM-head kernel that quantises a decode
// call's h rows itself, so that both produce the same codes and scales.
// ("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
// Agent-Driven", dense-GEMM section: W8A8 inputs quantised with
// round-to-nearest-even, identically on both sides.)
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace rlk {

// The scale of a row (or block) from its max |x|: the IEEE fp32 quotient
// amax / 448, and 1 for an all-zero row.
__device__ __forceinline__ float e4m3_scale(float amax) {
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}
// Scales at or above this take the reciprocal path of quotient<true>: a
// quotient that can reach a nonzero code then has a normal residual.
constexpr float kE4m3FastScaleMin = 0x1p-64f;

// x / sc rounded to nearest, from rs = the correctly rounded 1 / sc: the
// product's residual is exact under fma, and one correction step gives the
// correctly rounded quotient (Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", 1990).  The quotient has the sign of x
// whatever it rounds to, so the sign is copied from x: that keeps -0 for x = -0
// (the correction step alone gives +0 there) with one bit operation instead of
// a compare and a select (measured 4% faster for the weight).  Callers use it
// only while rs is finite and normal; the GPU tests check it against the IEEE
// division for every bf16 x and every scale amax/448 a bf16 amax can give.
__device__ __forceinline__ float div_by_scale(float x, float sc, float rs) {
    const float q = __fmul_rn(x, rs);
    const float e = __fmaf_rn(-q, sc, x);
    return copysignf(__fmaf_rn(e, rs, q), x);
}

template <bool kFast>
__device__ __forceinline__ float quotient(float x, float sc, float rs) {
    if constexpr (kFast)
        return div_by_scale(x, sc, rs);
    else
        return __fdiv_rn(x, sc);
}

template <bool kFast>
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float sc, float rs) {
    const uint32_t c0 = __nv_cvt_float_to_fp8(quotient<kFast>(a, sc, rs), __NV_SATFINITE, __NV_E4M3);
    const uint32_t c1 = __nv_cvt_float_to_fp8(quotient<kFast>(b, sc, rs), __NV_SATFINITE, __NV_E4M3);
    const uint32_t c2 = __nv_cvt_float_to_fp8(quotient<kFast>(c, sc, rs), __NV_SATFINITE, __NV_E4M3);
    const uint32_t c3 = __nv_cvt_float_to_fp8(quotient<kFast>(d, sc, rs), __NV_SATFINITE, __NV_E4M3);
    return c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
}

}  // namespace rlk
