/*
 * cbs_oracle.c -- CPU oracle for the fused Conv2d + BatchNorm + SiLU layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * GPU library is checked against.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or constant with the CUDA library under conv_bn_silu_gb300/csrc, and
 * it never includes or links it.
 *
 * What it computes (page 1, "YOLO26N Inference Optimisation", sections
 * "NHWC migration -- What NHWC is and why it matters" and "Weight layout";
 * page 3, "Edge optimisation of YOLO26", "Design notes" and "Highlights"):
 *
 *   z[n,co,oh,ow] = sum_{ci,r,s} x[n,ci,oh*S-P+r, ow*S-P+s] * w[co,ci,r,s]
 *                   (x is zero outside [0,H) x [0,W); NCHW input, OIHW weights)
 *   b = gamma * (z - mean) / sqrt(var + eps) + beta      (inference BatchNorm)
 *   y = b / (1 + exp(-b))                                (SiLU)
 *
 * The FP32 oracle keeps the three steps separate (no folding) and evaluates
 * every one of them in double; the result is rounded to float once at the end.
 *
 * The INT8 oracle follows the quantised scheme step by step in float
 * arithmetic with a fixed operation order (per-output-channel symmetric weight
 * scales, one activation scale, symmetric or with a zero point, integer
 * accumulation, bias folded in int32, SiLU in float, round-half-even back to
 * int8).  Its exp is our own
 * Cody-Waite range reduction (W. J. Cody and W. Waite, "Software Manual for
 * the Elementary Functions", 1980) followed by a degree-7 Taylor polynomial,
 * so that the result does not depend on any libm.  Build with
 * -ffp-contract=off so that no float expression is fused behind our back.
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py.
 */
#include <math.h>
#include <omp.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

ORACLE_API int oracle_out_dim(int in, int k, int stride, int pad)
{
    return (in + 2 * pad - k) / stride + 1;
}

/* Threads of the OpenMP loops below (for timing the oracle on one core or
 * on all of them). */
ORACLE_API void oracle_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
ORACLE_API int oracle_max_threads(void) { return omp_get_max_threads(); }

/* ---------------------------------------------------------------------- */
/* FP32 path: conv -> BN -> SiLU, each its own step, all in double.        */
/* ---------------------------------------------------------------------- */

/* Plain 7-loop convolution; z is [N, C_out, OH, OW] in double. */
ORACLE_API void oracle_conv2d(const float *x, const float *w, const float *conv_bias,
                              int N, int C_in, int H, int W, int C_out, int k,
                              int stride, int pad, double *z)
{
    const int OH = oracle_out_dim(H, k, stride, pad);
    const int OW = oracle_out_dim(W, k, stride, pad);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int n = 0; n < N; ++n) {
        for (int co = 0; co < C_out; ++co) {
            for (int oh = 0; oh < OH; ++oh) {
                for (int ow = 0; ow < OW; ++ow) {
                    double acc = conv_bias ? (double)conv_bias[co] : 0.0;
                    for (int ci = 0; ci < C_in; ++ci) {
                        for (int r = 0; r < k; ++r) {
                            const int ih = oh * stride - pad + r;
                            if (ih < 0 || ih >= H) continue;
                            for (int s = 0; s < k; ++s) {
                                const int iw = ow * stride - pad + s;
                                if (iw < 0 || iw >= W) continue;
                                const double xv = x[(((size_t)n * C_in + ci) * H + ih) * W + iw];
                                const double wv = w[(((size_t)co * C_in + ci) * k + r) * k + s];
                                acc += xv * wv;
                            }
                        }
                    }
                    z[(((size_t)n * C_out + co) * OH + oh) * OW + ow] = acc;
                }
            }
        }
    }
}

/* Inference BatchNorm with running statistics, in place on t [N, C, HW]. */
ORACLE_API void oracle_batchnorm(double *t, const float *gamma, const float *beta,
                                 const float *mean, const float *var, float eps,
                                 int N, int C, size_t HW)
{
#pragma omp parallel for collapse(2)
    for (int n = 0; n < N; ++n) {
        for (int c = 0; c < C; ++c) {
            const double g = gamma[c], b = beta[c], mu = mean[c];
            const double sd = sqrt((double)var[c] + (double)eps);
            double *p = t + ((size_t)n * C + c) * HW;
            for (size_t i = 0; i < HW; ++i) p[i] = g * (p[i] - mu) / sd + b;
        }
    }
}

/* SiLU(t) = t * sigmoid(t) = t / (1 + e^-t), in place. */
ORACLE_API void oracle_silu(double *t, size_t count)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) t[i] = t[i] / (1.0 + exp(-t[i]));
}

/* The whole FP32 layer: y (float, NCHW) = SiLU(BN(conv(x))).  `work` holds
 * N*C_out*OH*OW doubles and receives the unrounded result. */
ORACLE_API void oracle_conv_bn_silu_f32(const float *x, const float *w, const float *conv_bias,
                                        const float *gamma, const float *beta,
                                        const float *mean, const float *var, float eps,
                                        int N, int C_in, int H, int W, int C_out, int k,
                                        int stride, int pad, double *work, float *y)
{
    const int OH = oracle_out_dim(H, k, stride, pad);
    const int OW = oracle_out_dim(W, k, stride, pad);
    const size_t HW = (size_t)OH * OW, total = (size_t)N * C_out * HW;
    oracle_conv2d(x, w, conv_bias, N, C_in, H, W, C_out, k, stride, pad, work);
    oracle_batchnorm(work, gamma, beta, mean, var, eps, N, C_out, HW);
    oracle_silu(work, total);
    for (size_t i = 0; i < total; ++i) y[i] = (float)work[i];
}

/* Conv -> BN -> activation -> + residual, the plain conv + bias and residual
 * forms beside the fused layer in the kernel profile of "YOLO26N Inference
 * Optimisation" (conv2d_forward, elemwise_add):
 *   y = act(BN(conv(x))) + r,   act = SiLU (act == 0) or identity (act == 1),
 * r an NCHW float tensor shaped like y, or NULL for none.  Same order of
 * steps as oracle_conv_bn_silu_f32, double arithmetic, rounded once. */
ORACLE_API void oracle_conv_bn_act_f32(const float *x, const float *w, const float *conv_bias,
                                       const float *gamma, const float *beta,
                                       const float *mean, const float *var, float eps,
                                       int N, int C_in, int H, int W, int C_out, int k,
                                       int stride, int pad, int act, const float *residual,
                                       double *work, float *y)
{
    const int OH = oracle_out_dim(H, k, stride, pad);
    const int OW = oracle_out_dim(W, k, stride, pad);
    const size_t total = (size_t)N * C_out * OH * OW;
    oracle_conv2d(x, w, conv_bias, N, C_in, H, W, C_out, k, stride, pad, work);
    oracle_batchnorm(work, gamma, beta, mean, var, eps, N, C_out, (size_t)OH * OW);
    if (act == 0) oracle_silu(work, total);
    if (residual)
        for (size_t i = 0; i < total; ++i) work[i] += (double)residual[i];
    for (size_t i = 0; i < total; ++i) y[i] = (float)work[i];
}

/* ---------------------------------------------------------------------- */
/* Glue beside the convolutions: max pooling.                              */
/* ---------------------------------------------------------------------- */

/* 2-D max pooling ("YOLO26N Inference Optimisation", kernel profile and "Op-by-op
 * impact": maxpool2d, three per frame): y[n,c,oh,ow] = max over the k x k
 * window at (oh*S-P, ow*S-P) of the positions inside the image (padding
 * takes no part); OH = (H + 2P - k)/S + 1 (floor).  A NaN in the window
 * gives NaN.  x, y: NCHW float. */
ORACLE_API void oracle_maxpool2d_f32(const float *x, int N, int C, int H, int W, int k, int stride, int pad,
                                     float *y)
{
    const int OH = oracle_out_dim(H, k, stride, pad);
    const int OW = oracle_out_dim(W, k, stride, pad);
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C; ++c)
            for (int oh = 0; oh < OH; ++oh)
                for (int ow = 0; ow < OW; ++ow) {
                    float m = -INFINITY;
                    int nan = 0;
                    for (int r = 0; r < k; ++r) {
                        const int ih = oh * stride - pad + r;
                        if (ih < 0 || ih >= H) continue;
                        for (int s = 0; s < k; ++s) {
                            const int iw = ow * stride - pad + s;
                            if (iw < 0 || iw >= W) continue;
                            const float v = x[(((size_t)n * C + c) * H + ih) * W + iw];
                            if (v != v) nan = 1;
                            else if (v > m) m = v;
                        }
                    }
                    y[(((size_t)n * C + c) * OH + oh) * OW + ow] = nan ? NAN : m;
                }
}

/* ---------------------------------------------------------------------- */
/* INT8 path.                                                              */
/* ---------------------------------------------------------------------- */

/* Round half to even to an integer-valued float (default rounding mode). */
static float rne(float v) { return nearbyintf(v); }

/* Our exp for the INT8 epilogue (Cody-Waite reduction, Taylor degree 7).
 *   k = nearest integer to x * log2(e)
 *   r = x - k*ln2, with ln2 split in a 16-bit head and a float tail
 *   e^r ~ sum_{n<=7} r^n / n!   (Horner, fused multiply-adds)
 *   e^x = e^r * 2^k             (2^k built from its exponent bits)
 * Out of range: x > 88 gives +inf, x < -87 gives +0. */
static const float CW_LOG2E  = 0x1.715476p+0f;   /* float(1/ln 2)            */
static const float CW_LN2_HI = 0x1.62e4p-1f;     /* ln 2 truncated to 16 bits */
static const float CW_LN2_LO = 0x1.7f7d1cp-20f;  /* float(ln 2 - CW_LN2_HI)   */

ORACLE_API float oracle_spec_exp(float x)
{
    if (x > 88.0f) { const uint32_t b = 0x7f800000u; float f; memcpy(&f, &b, 4); return f; }
    if (x < -87.0f) return 0.0f;
    const float kf = rne(x * CW_LOG2E);
    float r = fmaf(-kf, CW_LN2_HI, x);
    r = fmaf(-kf, CW_LN2_LO, r);
    /* Taylor coefficients 1/n!, n = 7 .. 0, each rounded to float. */
    float p = 0x1.a01a02p-13f;           /* 1/5040 */
    p = fmaf(p, r, 0x1.6c16c2p-10f);     /* 1/720  */
    p = fmaf(p, r, 0x1.111112p-7f);      /* 1/120  */
    p = fmaf(p, r, 0x1.555556p-5f);      /* 1/24   */
    p = fmaf(p, r, 0x1.555556p-3f);      /* 1/6    */
    p = fmaf(p, r, 0.5f);                /* 1/2    */
    p = fmaf(p, r, 1.0f);                /* 1/1    */
    p = fmaf(p, r, 1.0f);                /* 1/0!   */
    const int k = (int)kf;               /* in [-126, 127] here */
    const uint32_t bits = (uint32_t)(k + 127) << 23;
    float scale; memcpy(&scale, &bits, 4);
    return p * scale;
}

ORACLE_API void oracle_spec_exp_array(const float *x, float *y, size_t count)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) y[i] = oracle_spec_exp(x[i]);
}

/* Activation quantisation: q = clamp(rne(x / s_x), -128, 127). */
ORACLE_API void oracle_quantize_act(const float *x, size_t count, float s_x, int8_t *q)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) {
        float v = x[i] / s_x;
        v = v < -128.0f ? -128.0f : (v > 127.0f ? 127.0f : v);
        q[i] = (int8_t)rne(v);
    }
}

/* Asymmetric activation quantisation ("Edge optimisation of YOLO26", Design
 * notes: asymmetric activations, symmetric weights; the affine scheme of
 * Jacob et al., CVPR 2018, r = s (q - z)), on signed 8-bit codes:
 *   q = clamp(rne(x / s_x) + z_x, -128, 127),   z_x in [-128, 127].
 * A uint8 code u with zero point z_u is the same value as q = u - 128 with
 * z = z_u - 128.  With z_x = 0 this is oracle_quantize_act. */
ORACLE_API void oracle_quantize_act_zp(const float *x, size_t count, float s_x, int z_x, int8_t *q)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) {
        float v = rne(x[i] / s_x) + (float)z_x;
        v = v < -128.0f ? -128.0f : (v > 127.0f ? 127.0f : v);
        q[i] = (int8_t)v;
    }
}

/* Largest relative error of oracle_spec_exp against the double-precision
 * exp over every float x in [lo, hi] (walked by bit pattern): the bound an
 * error analysis of the INT8 epilogue may rely on. */
ORACLE_API double oracle_spec_exp_max_rel_err(float lo, float hi)
{
    /* Floats in [lo, hi] in increasing order, mapped to a monotone integer key. */
    uint32_t ulo, uhi;
    memcpy(&ulo, &lo, 4);
    memcpy(&uhi, &hi, 4);
    const int64_t klo = (ulo & 0x80000000u) ? -(int64_t)(ulo & 0x7fffffffu) : (int64_t)ulo;
    const int64_t khi = (uhi & 0x80000000u) ? -(int64_t)(uhi & 0x7fffffffu) : (int64_t)uhi;
    double worst = 0.0;
#pragma omp parallel for reduction(max : worst) schedule(static)
    for (int64_t k = klo; k <= khi; ++k) {
        const uint32_t u = k < 0 ? (0x80000000u | (uint32_t)(-k)) : (uint32_t)k;
        float x;
        memcpy(&x, &u, 4);
        const double ref = exp((double)x);
        const double err = fabs((double)oracle_spec_exp(x) - ref) / ref;
        if (err > worst) worst = err;
    }
    return worst;
}

/* Dequantisation at a seam between an INT8 layer and a layer kept in float
 * ("Edge optimisation of YOLO26", Highlights: sensitive layers are kept in
 * float; the affine scheme r = s (q - z) of Jacob et al., CVPR 2018):
 *   r = (float)(q - z) * s,   one float multiply (q - z is exact in float). */
ORACLE_API void oracle_dequantize_i8(const int8_t *q, size_t count, float s, int z, float *r)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) r[i] = (float)((int)q[i] - z) * s;
}

/* Round to bfloat16 (the upper 16 bits of the float), to nearest with ties
 * to even, and return the rounded value as float: the format in which a
 * layer kept in BF16 receives its input.  NaN stays NaN. */
ORACLE_API void oracle_round_bf16(const float *x, size_t count, float *out)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) {
        uint32_t u;
        memcpy(&u, &x[i], 4);
        if ((u & 0x7fffffffu) > 0x7f800000u) {
            u |= 0x00400000u;            /* quiet NaN */
        } else {
            const uint32_t rest = u & 0xffffu, keep = u >> 16;
            /* above half an ulp, or exactly half with an odd kept part: round up */
            if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) u = (keep + 1u) << 16;
            else u = keep << 16;
        }
        u &= 0xffff0000u;
        memcpy(&out[i], &u, 4);
    }
}

/* Fold BN into the weights and quantise them per output channel.
 *   s_c   = gamma / sqrtf(var + eps)
 *   w'    = w * s_c                      b' = beta - mean * s_c
 *   s_w   = max_i |w'[c,i]| / 127        (s_w = 1 when the channel is all zero)
 *   q_w   = rne(w' / s_w)                (in [-127, 127])
 *   m_c   = s_x * s_w
 *   b_i32 = rne(b' / m_c), saturated to the int32 range.
 * w, q_w: [C_out][KK] with KK = C_in*k*k (OIHW order). */
ORACLE_API void oracle_fold_quant_i8(const float *w, const float *gamma, const float *beta,
                                     const float *mean, const float *var, float eps, float s_x,
                                     int C_out, int KK, int8_t *q_w, int32_t *bias_i32, float *m_c)
{
    for (int c = 0; c < C_out; ++c) {
        const float s_c = gamma[c] / sqrtf(var[c] + eps);
        float amax = 0.0f;
        for (int i = 0; i < KK; ++i) {
            const float wf = w[(size_t)c * KK + i] * s_c;
            const float a = fabsf(wf);
            if (a > amax) amax = a;
        }
        float s_w = amax / 127.0f;
        if (s_w == 0.0f) s_w = 1.0f;
        for (int i = 0; i < KK; ++i) {
            const float wf = w[(size_t)c * KK + i] * s_c;
            float v = rne(wf / s_w);
            v = v < -127.0f ? -127.0f : (v > 127.0f ? 127.0f : v);
            q_w[(size_t)c * KK + i] = (int8_t)v;
        }
        const float mc = s_x * s_w;
        const float prod = mean[c] * s_c;
        const float bf = beta[c] - prod;
        const float bq = rne(bf / mc);
        int32_t bi;
        if (bq >= 2147483648.0f) bi = INT32_MAX;
        else if (bq < -2147483648.0f) bi = INT32_MIN;
        else bi = (int32_t)bq;
        bias_i32[c] = bi;
        m_c[c] = mc;
    }
}

/* Requantising epilogue for one accumulator value:
 *   t = float(acc) * m_c;  u = t / (1 + exp(-t));  v = u * (1 / s_y);
 *   q = rne(clamp(v, -128, 127)). */
ORACLE_API int8_t oracle_requant(int32_t acc, float m_c, float inv_s_y)
{
    const float t = (float)acc * m_c;
    const float e = oracle_spec_exp(-t);
    const float u = t / (1.0f + e);
    float v = u * inv_s_y;
    v = v < -128.0f ? -128.0f : (v > 127.0f ? 127.0f : v);
    return (int8_t)rne(v);
}

/* Requantisation to an asymmetric output code:
 *   t = float(acc) * m_c;  u = t / (1 + exp(-t));  v = u * (1 / s_y);
 *   q = clamp(rne(v) + z_y, -128, 127).
 * With z_y = 0 this is oracle_requant (the bounds are integers). */
ORACLE_API int8_t oracle_requant_zp(int32_t acc, float m_c, float inv_s_y, int z_y)
{
    const float t = (float)acc * m_c;
    const float e = oracle_spec_exp(-t);
    const float u = t / (1.0f + e);
    float v = rne(u * inv_s_y) + (float)z_y;
    v = v < -128.0f ? -128.0f : (v > 127.0f ? 127.0f : v);
    return (int8_t)v;
}

/* oracle_requant_zp over arrays of accumulators and scales (one output each). */
ORACLE_API void oracle_requant_zp_array(const int32_t *acc, const float *m_c, size_t count, float inv_s_y, int z_y,
                                        int8_t *q)
{
#pragma omp parallel for
    for (size_t i = 0; i < count; ++i) q[i] = oracle_requant_zp(acc[i], m_c[i], inv_s_y, z_y);
}

/* INT8 layer: integer convolution (int64 accumulation; the sum must fit in
 * int32, which the function checks), plus the int32 bias, then the epilogue.
 * q_x: [N][C_in][H][W], q_w: [C_out][C_in][k][k], q_y: [N][C_out][OH][OW].
 * acc_out (nullable) receives the int32 accumulators including the bias.
 * Returns 0, or -1 if an accumulator left the int32 range. */
ORACLE_API int oracle_conv_i8(const int8_t *q_x, const int8_t *q_w, const int32_t *bias_i32,
                              const float *m_c, float s_y, int N, int C_in, int H, int W,
                              int C_out, int k, int stride, int pad, int8_t *q_y, int32_t *acc_out)
{
    const int OH = oracle_out_dim(H, k, stride, pad);
    const int OW = oracle_out_dim(W, k, stride, pad);
    const float inv_s_y = 1.0f / s_y;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(|:bad)
    for (int n = 0; n < N; ++n) {
        for (int co = 0; co < C_out; ++co) {
            for (int oh = 0; oh < OH; ++oh) {
                for (int ow = 0; ow < OW; ++ow) {
                    int64_t acc = bias_i32[co];
                    for (int ci = 0; ci < C_in; ++ci) {
                        for (int r = 0; r < k; ++r) {
                            const int ih = oh * stride - pad + r;
                            if (ih < 0 || ih >= H) continue;
                            for (int s = 0; s < k; ++s) {
                                const int iw = ow * stride - pad + s;
                                if (iw < 0 || iw >= W) continue;
                                acc += (int64_t)q_x[(((size_t)n * C_in + ci) * H + ih) * W + iw] *
                                       (int64_t)q_w[(((size_t)co * C_in + ci) * k + r) * k + s];
                            }
                        }
                    }
                    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
                    const size_t o = (((size_t)n * C_out + co) * OH + oh) * OW + ow;
                    if (acc_out) acc_out[o] = (int32_t)acc;
                    q_y[o] = oracle_requant((int32_t)acc, m_c[co], inv_s_y);
                }
            }
        }
    }
    return bad ? -1 : 0;
}

/* The INT8 layer with asymmetric activations: input codes q_x with zero point
 * z_x, output codes with zero point z_y, symmetric per-channel weights.
 *   acc = bias_i32 + sum over the taps inside the image of (q_x - z_x) * q_w
 * (a tap outside the image is a real zero and adds nothing), then
 * oracle_requant_zp.  Layouts, acc_out and the return value as for
 * oracle_conv_i8; with z_x = z_y = 0 the two functions agree. */
ORACLE_API int oracle_conv_i8_zp(const int8_t *q_x, const int8_t *q_w, const int32_t *bias_i32,
                                 const float *m_c, float s_y, int z_x, int z_y, int N, int C_in, int H, int W,
                                 int C_out, int k, int stride, int pad, int8_t *q_y, int32_t *acc_out)
{
    const int OH = oracle_out_dim(H, k, stride, pad);
    const int OW = oracle_out_dim(W, k, stride, pad);
    const float inv_s_y = 1.0f / s_y;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(|:bad)
    for (int n = 0; n < N; ++n) {
        for (int co = 0; co < C_out; ++co) {
            for (int oh = 0; oh < OH; ++oh) {
                for (int ow = 0; ow < OW; ++ow) {
                    int64_t acc = bias_i32[co];
                    for (int ci = 0; ci < C_in; ++ci) {
                        for (int r = 0; r < k; ++r) {
                            const int ih = oh * stride - pad + r;
                            if (ih < 0 || ih >= H) continue;
                            for (int s = 0; s < k; ++s) {
                                const int iw = ow * stride - pad + s;
                                if (iw < 0 || iw >= W) continue;
                                const int64_t xv = (int64_t)q_x[(((size_t)n * C_in + ci) * H + ih) * W + iw] - z_x;
                                acc += xv * (int64_t)q_w[(((size_t)co * C_in + ci) * k + r) * k + s];
                            }
                        }
                    }
                    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
                    const size_t o = (((size_t)n * C_out + co) * OH + oh) * OW + ow;
                    if (acc_out) acc_out[o] = (int32_t)acc;
                    q_y[o] = oracle_requant_zp((int32_t)acc, m_c[co], inv_s_y, z_y);
                }
            }
        }
    }
    return bad ? -1 : 0;
}
