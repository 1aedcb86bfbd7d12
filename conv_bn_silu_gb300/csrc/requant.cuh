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

// The same code through the hardware approximations where that is provably
// the same result.  With t = float(acc) * m_c (identical in both) and
// |t| <= 80, w = t * rcp(1 + ex2(-t log2 e)) * inv_s_y differs from the
// specified value (before rounding) by less than
//   |w| (f (1.5e-6 + 2.4e-7 |t|) + 1.2e-6),   f = min(1, 1.001 ex2(-t log2 e)),
// which is twice the first-order error of the two evaluations when the
// specified exp is within 1.2e-7 relative, ex2.approx within 4.8e-7 and
// rcp.approx within 2.4e-7 over this range (each of these bounds is
// measured exhaustively by the tests).  When w is farther than that from
// every half-integer both round to the same integer, and the zero point and
// the clamp are the same steps; otherwise, and for |t| > 80, the specified
// steps run.  About one value in a few thousand takes that path.
static __device__ __forceinline__ int requant_i8_fast(int acc, float m_c, float inv_s_y, int z_y = 0) {
    const float t = __fmul_rn(__int2float_rn(acc), m_c);
    if (fabsf(t) <= 80.0f) {
        float e, r;
        const float y = __fmul_rn(t, -1.44269502f);   // -t log2(e)
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(y));
        const float d = __fadd_rn(1.0f, e);
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
        const float w = __fmul_rn(__fmul_rn(t, r), inv_s_y);
        const float k = rintf(w);
        const float dist = __fsub_rn(0.5f, fabsf(__fsub_rn(w, k)));   // distance to the nearest half-integer
        const float f = fminf(1.0f, __fmul_rn(e, 1.001f));
        const float bound = __fmul_rn(fabsf(w), __fmaf_rn(f, __fmaf_rn(2.4e-7f, fabsf(t), 1.5e-6f), 1.2e-6f));
        if (dist > bound) {
            float v = __fadd_rn(k, (float)z_y);
            v = fminf(fmaxf(v, -128.0f), 127.0f);
            return (int)v;
        }
    }
    return requant_i8(acc, m_c, inv_s_y, z_y);
}

}  // namespace cbs
