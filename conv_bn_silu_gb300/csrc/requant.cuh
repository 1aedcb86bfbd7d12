// requant.cuh -- the INT8 requantising epilogue, specified bit for bit
// (page 3, "Edge optimisation of YOLO26", "Highlights": SiLU in float, then
// round half to even back to int8).  Shared by the library's INT8 kernels.
#pragma once

namespace cbs {

// Our exp for the requantising epilogue, specified bit for bit:
// Cody-Waite reduction with a 16-bit head of ln 2, degree-7 Taylor
// polynomial in Horner form with fused multiply-adds, scaling by 2^k through
// the exponent field; +inf above 88, +0 below -87.
static __device__ __forceinline__ float cw_exp(float x) {
    if (x > 88.0f) return __int_as_float(0x7f800000);
    if (x < -87.0f) return 0.0f;
    const float kf = rintf(__fmul_rn(x, 0x1.715476p+0f));
    float r = __fmaf_rn(-kf, 0x1.62e4p-1f, x);
    r = __fmaf_rn(-kf, 0x1.7f7d1cp-20f, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int k = (int)kf;
    return __fmul_rn(p, __int_as_float((k + 127) << 23));
}

// q = clamp(rne(SiLU(float(acc) * m_c) * inv_s_y) + z_y, -128, 127), IEEE
// steps.  With z_y = 0 this is rne(clamp(v, -128, 127)): the bounds are
// integers, so rounding and clamping commute.
static __device__ __forceinline__ int requant_i8(int acc, float m_c, float inv_s_y, int z_y = 0) {
    const float t = __fmul_rn(__int2float_rn(acc), m_c);
    const float e = cw_exp(-t);
    const float u = __fdiv_rn(t, __fadd_rn(1.0f, e));
    float v = __fadd_rn(rintf(__fmul_rn(u, inv_s_y)), (float)z_y);
    v = fminf(fmaxf(v, -128.0f), 127.0f);
    return (int)v;
}

}  // namespace cbs
