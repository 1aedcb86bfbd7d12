// k_stem.cu -- direct convolution for layers with at most four input channels
// (the YOLO26n stem: 3 -> 16 channels, 3x3, stride 2, on the 640x640 frame).
//
// With three input channels the implicit GEMM's K is 27: padding it to a
// tensor-core K step would move 5x the real activation bytes through shared
// memory for a layer that is bound by memory and FMA issue, not by MMA.  Here
// each thread computes one output pixel for every output channel directly,
// reading its 3x3xC window (neighbouring threads share it through L1) and the
// folded weights from shared memory, with FP32 fused multiply-adds (exact
// integer sums for INT8).  The epilogue is the same as the other variants':
// + folded bias, SiLU, store (or the specified INT8 requantisation).
#include <cuda_bf16.h>

#include "cbs_internal.cuh"
#include "requant.cuh"

namespace cbs {
namespace {

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f<int8_t>(int8_t v) { return (float)v; }

// Output pixels per thread: every weight read from shared memory feeds
// P x 4 multiply-adds.  Measured on GB300 for the 3 -> 16 stem: FP32 is
// fastest at one pixel per thread (more warps hide the scalar NCHW loads),
// BF16 at two, INT8 (integer multiply-adds) at four.
template <int KIND, int COUT>
struct StemTile {
    static constexpr int P = KIND == 0 ? 1 : KIND == 1 ? (COUT <= 32 ? 2 : 1) : (COUT <= 16 ? 4 : (COUT <= 32 ? 2 : 1));
};

// Stores one output pixel: 16-byte vectors when an NHWC pixel holds exactly
// the register tile's channels, else one element per channel.
template <int KIND, int COUT, bool OUT_NHWC>
__device__ __forceinline__ void store_pixel(const StemLaunch &a, long long pix, int img, int oh, int ow,
                                            float (&of)[COUT], const int (&oq)[COUT]) {
    // Residual (float kinds): the same element of r, added after the activation.
    const size_t plane = (size_t)a.OH * a.out_row_stride;
    const size_t opix = (size_t)oh * a.out_row_stride + ow;
    if (KIND != 2 && a.residual) {
#pragma unroll
        for (int c = 0; c < COUT; ++c) {
            if (c >= a.Cout) break;
            const size_t off = OUT_NHWC ? (size_t)pix * a.Cout + c : ((size_t)img * a.Cout + c) * plane + opix;
            of[c] += KIND == 0 ? static_cast<const float *>(a.residual)[off]
                               : __bfloat162float(static_cast<const __nv_bfloat16 *>(a.residual)[off]);
        }
    }
    if (OUT_NHWC && a.Cout == COUT) {
        if (KIND == 0) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.y) + (size_t)pix * COUT);
#pragma unroll
            for (int c = 0; c < COUT / 4; ++c) dst[c] = make_float4(of[4 * c], of[4 * c + 1], of[4 * c + 2], of[4 * c + 3]);
        } else if (KIND == 1) {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.y) + (size_t)pix * COUT);
#pragma unroll
            for (int c = 0; c < COUT / 8; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(of[8 * c + 2 * k], of[8 * c + 2 * k + 1]);
                    w[k] = *reinterpret_cast<uint32_t *>(&h2);
                }
                dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<int8_t *>(a.y) + (size_t)pix * COUT);
#pragma unroll
            for (int c = 0; c < COUT / 16; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    w[k] = (uint32_t)(uint8_t)oq[16 * c + 4 * k] | ((uint32_t)(uint8_t)oq[16 * c + 4 * k + 1] << 8) |
                           ((uint32_t)(uint8_t)oq[16 * c + 4 * k + 2] << 16) |
                           ((uint32_t)(uint8_t)oq[16 * c + 4 * k + 3] << 24);
                dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < COUT; ++c) {
        if (c >= a.Cout) break;
        const size_t off = OUT_NHWC ? (size_t)pix * a.Cout + c : ((size_t)img * a.Cout + c) * plane + opix;
        if (KIND == 2)
            static_cast<int8_t *>(a.y)[off] = (int8_t)oq[c];
        else if (KIND == 0)
            static_cast<float *>(a.y)[off] = of[c];
        else
            static_cast<__nv_bfloat16 *>(a.y)[off] = __float2bfloat16_rn(of[c]);
    }
}

// KIND: 0 float in/out, 1 bf16 in/out, 2 int8 in/out (requantised).
template <int KIND, int COUT, bool IN_NHWC, bool OUT_NHWC>
__global__ void __launch_bounds__(256) stem_kernel(const StemLaunch a) {
    using Tin = typename std::conditional<KIND == 0, float, typename std::conditional<KIND == 1, __nv_bfloat16, int8_t>::type>::type;
    constexpr int P = StemTile<KIND, COUT>::P;
    extern __shared__ float4 wsm4[];  // [KK * c_pad][COUT] floats
    float *wsm = reinterpret_cast<float *>(wsm4);
    const int KK = a.KS * a.KS;
    const int kpad = KK * a.c_pad;
    // Folded weights: packed [C_out][KK * c_pad] (float, or bf16 holding
    // bf16 values / int8 codes) -> [tap * c_pad + ci][co] as float.
    for (int idx = threadIdx.x; idx < kpad * COUT; idx += blockDim.x) {
        const int co = idx / kpad, k = idx - co * kpad;
        float v = 0.0f;
        if (co < a.Cout) {
            if (KIND == 0)
                v = static_cast<const float *>(a.w)[(size_t)co * kpad + k];
            else
                v = __bfloat162float(static_cast<const __nv_bfloat16 *>(a.w)[(size_t)co * kpad + k]);
        }
        wsm[k * COUT + co] = v;
    }
    __syncthreads();

    const long long total = (long long)a.N * a.OH * a.OW;
    const long long pix0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * P;
    if (pix0 >= total) return;
    const int ohw = a.OH * a.OW;
    int img[P], oh[P], ow[P];
    bool live[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        const long long pix = pix0 + j;
        live[j] = pix < total;
        const long long pc = live[j] ? pix : pix0;
        img[j] = (int)(pc / ohw);
        const int rem = (int)(pc - (long long)img[j] * ohw);
        oh[j] = rem / a.OW;
        ow[j] = rem - oh[j] * a.OW;
    }
    const Tin *x = static_cast<const Tin *>(a.x);

    float accf[P][COUT];
#pragma unroll
    for (int j = 0; j < P; ++j)
#pragma unroll
        for (int c = 0; c < COUT; ++c) accf[j][c] = 0.0f;

    const bool vec_in = IN_NHWC && a.c_pad == 4;  // one 4-channel vector load per tap
    for (int r = 0; r < a.KS; ++r) {
        for (int s = 0; s < a.KS; ++s) {
            const float *wt = wsm + (r * a.KS + s) * a.c_pad * COUT;
            // The tap's input channels of each pixel (zero outside the image).
            float xf[P][4];
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const int ih = oh[j] * a.stride - a.pad + r;
                const int iw = ow[j] * a.stride - a.pad + s;
                const bool in = live[j] && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;
                Tin xv[4];
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) xv[ci] = Tin(0);
                if (in) {
                    if (vec_in) {
                        const Tin *src = x + (((size_t)img[j] * a.H + ih) * a.W + iw) * 4;
                        if (KIND == 0) {
                            const float4 q = *reinterpret_cast<const float4 *>(src);
                            xv[0] = q.x; xv[1] = q.y; xv[2] = q.z; xv[3] = q.w;
                        } else if (KIND == 1) {
                            const uint2 q = *reinterpret_cast<const uint2 *>(src);
                            const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&q.x);
                            const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&q.y);
                            xv[0] = lo.x; xv[1] = lo.y; xv[2] = hi.x; xv[3] = hi.y;
                        } else {
                            const int q = *reinterpret_cast<const int *>(src);
                            xv[0] = (int8_t)(q & 0xff); xv[1] = (int8_t)((q >> 8) & 0xff);
                            xv[2] = (int8_t)((q >> 16) & 0xff); xv[3] = (int8_t)(q >> 24);
                        }
                    } else {
#pragma unroll
                        for (int ci = 0; ci < 4; ++ci) {
                            if (ci >= a.C) break;
                            xv[ci] = IN_NHWC ? x[(((size_t)img[j] * a.H + ih) * a.W + iw) * a.c_pad + ci]
                                             : x[(((size_t)img[j] * a.C + ci) * a.H + ih) * a.W + iw];
                        }
                    }
                }
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) xf[j][ci] = to_f<Tin>(xv[ci]);
            }
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
                if (ci >= a.C) break;
                const float4 *w4 = reinterpret_cast<const float4 *>(wt + ci * COUT);
#pragma unroll
                for (int c = 0; c < COUT / 4; ++c) {
                    const float4 w = w4[c];
                    // INT8 too: codes are exact in float, every product
                    // |q_x q_w| <= 16256 and a sum of at most 7*7*4 = 196 of
                    // them stays below 2^24, so the float accumulation is the
                    // exact integer sum (and runs at the FMA rate, twice IMAD's).
#pragma unroll
                    for (int j = 0; j < P; ++j) {
                        accf[j][4 * c] = fmaf(xf[j][ci], w.x, accf[j][4 * c]);
                        accf[j][4 * c + 1] = fmaf(xf[j][ci], w.y, accf[j][4 * c + 1]);
                        accf[j][4 * c + 2] = fmaf(xf[j][ci], w.z, accf[j][4 * c + 2]);
                        accf[j][4 * c + 3] = fmaf(xf[j][ci], w.w, accf[j][4 * c + 3]);
                    }
                }
            }
        }
    }

    // Epilogue: + bias, SiLU (or the INT8 requantisation), then stores; an
    // NHWC pixel whose channel count is the register tile's is written with
    // 16-byte vector stores (the P pixels of a thread are contiguous).
    float bias_f[COUT];
    int bias_i[COUT];
    float mc[COUT];
#pragma unroll
    for (int c = 0; c < COUT; ++c) {
        const bool lc = c < a.Cout;
        bias_f[c] = (KIND != 2 && lc) ? static_cast<const float *>(a.bias)[c] : 0.0f;
        bias_i[c] = (KIND == 2 && lc) ? static_cast<const int32_t *>(a.bias)[c] : 0;
        mc[c] = (KIND == 2 && lc) ? a.m_c[c] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < P; ++j) {
        if (!live[j]) continue;
        const long long pix = pix0 + j;
        float of[COUT];
        int oq[COUT];
#pragma unroll
        for (int c = 0; c < COUT; ++c) {
            if (KIND == 2)
                oq[c] = c < a.Cout ? requant_i8(__float2int_rn(accf[j][c]) + bias_i[c], mc[c], a.inv_s_y) : 0;
            else
                of[c] = a.act == CBS_ACT_IDENTITY ? accf[j][c] + bias_f[c] : silu_fast(accf[j][c] + bias_f[c]);
        }
        store_pixel<KIND, COUT, OUT_NHWC>(a, pix, img[j], oh[j], ow[j], of, oq);
    }
}

template <int KIND, int COUT>
cudaError_t launch_kind(const StemLaunch &L, cudaStream_t s) {
    const long long total = (long long)L.N * L.OH * L.OW;
    constexpr int P = StemTile<KIND, COUT>::P;
    const int grid = (int)((total + 256 * P - 1) / (256 * P));
    const int smem = L.KS * L.KS * L.c_pad * COUT * (int)sizeof(float);
    if (smem > 48 * 1024) {  // 7x7 filters with 64 output channels need 49 KB of weights
        cudaError_t e;
        if (L.in_nhwc && L.out_nhwc) e = set_max_dyn_smem(stem_kernel<KIND, COUT, true, true>, smem);
        else if (L.in_nhwc) e = set_max_dyn_smem(stem_kernel<KIND, COUT, true, false>, smem);
        else if (L.out_nhwc) e = set_max_dyn_smem(stem_kernel<KIND, COUT, false, true>, smem);
        else e = set_max_dyn_smem(stem_kernel<KIND, COUT, false, false>, smem);
        if (e != cudaSuccess) return e;
    }
    if (L.in_nhwc && L.out_nhwc) stem_kernel<KIND, COUT, true, true><<<grid, 256, smem, s>>>(L);
    else if (L.in_nhwc) stem_kernel<KIND, COUT, true, false><<<grid, 256, smem, s>>>(L);
    else if (L.out_nhwc) stem_kernel<KIND, COUT, false, true><<<grid, 256, smem, s>>>(L);
    else stem_kernel<KIND, COUT, false, false><<<grid, 256, smem, s>>>(L);
    return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_cout(const StemLaunch &L, cudaStream_t s) {
    if (L.Cout <= 16) return launch_kind<KIND, 16>(L, s);
    if (L.Cout <= 32) return launch_kind<KIND, 32>(L, s);
    return launch_kind<KIND, 64>(L, s);
}

}  // namespace

cudaError_t launch_stem(const StemLaunch &L, cudaStream_t s) {
    if (L.N == 0) return cudaSuccess;
    switch (L.kind) {
        case 0: return launch_cout<0>(L, s);
        case 1: return launch_cout<1>(L, s);
        case 2: return launch_cout<2>(L, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace cbs
