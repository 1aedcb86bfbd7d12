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
#include <algorithm>
#include <cuda_bf16.h>

#include "cbs_internal.cuh"
#include "requant.cuh"
#include "tc_ptx.cuh"

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
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
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
                // Outside the image the input is a real zero: code 0, or for
                // INT8 the code of zero, z_x.  (With an input zero point the
                // fold's bias is bias_i32 - z_x * sum(q_w), so every tap then
                // contributes (q - z_x) * q_w, inside the image or not.)
                Tin xv[4];
#pragma unroll
                for (int ci = 0; ci < 4; ++ci) xv[ci] = KIND == 2 ? Tin(a.zp_x) : Tin(0);
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
                oq[c] = c < a.Cout ? requant_i8_fast((int)((unsigned)__float2int_rn(accf[j][c]) + (unsigned)bias_i[c]),
                                                mc[c], a.inv_s_y, a.zp_y)
                                   : 0;
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
    // Plain launches, as for the CUDA-core implicit GEMM (see k_simt.cu).
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

namespace {

// ------------------------------------------------------ tensor-core stem
// BF16 stems with 4-channel NHWC pixels and k <= 3: the contraction is an
// M x 16..64 x K<=48 GEMM, one M=128 tile per 128 output pixels.  Persistent
// CTAs of 256 threads each keep the weights (B) in shared memory and walk
// their tiles with a ring of kStemTcStages A tiles.  Threads t and t + 128
// share output pixel t of a tile (TMEM lane t):
//   - each gathers half of the pixel's taps into row t of a 128-byte-swizzled
//     A tile with cp.async (zero-filled outside the image), kStemTcStages - 1
//     tiles ahead of the MMA;
//   - one thread issues the tile's MMAs into one of two TMEM accumulators
//     and commits them to that accumulator's mbarrier;
//   - while tile i's MMAs run, each thread reads alternate 8-channel groups of
//     tile i-1's accumulator back for bias, activation, residual and stores.
// K layout.  In general row t holds tap s (4 channels, 8 bytes) at byte 8s.
// For 3x3, stride 2, pad 1 and an even input width the row instead holds, for
// each kernel row r, the two 16-byte pixel pairs starting at input column
// 2*ow-2: four pixels of which the first is unused (its slot is zeroed after
// the copy lands and its weights are zero), so each pixel takes six aligned
// 16-byte copies instead of nine 8-byte ones.
constexpr uint64_t kStemWaitNs = 2000000000ull;

// n / d for 0 <= n < 2^31 as (umulhi(n, m) + n) >> l, the round-up
// multiplier of Granlund and Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994): l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
struct FastDiv {
    uint32_t m, l;
};

FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{(uint32_t)m, l};
}

__device__ __forceinline__ int fast_div(int n, FastDiv f) {
    return (int)((__umulhi((uint32_t)n, f.m) + (uint32_t)n) >> f.l);
}

struct StemTcGeom {
    int total;          // output pixels (< 2^31 - 128)
    int n_tiles;        // 128-pixel tiles
    FastDiv div_ohw;    // by OH * OW
    FastDiv div_ow;     // by OW
};

// SiLU as h + h tanh(h), h = z / 2 (sigma(z) = (1 + tanh(z / 2)) / 2).
__device__ __forceinline__ float silu_tanh(float h) {
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(h));
    return fmaf(h, th, h);
}

// Two floats rounded to bf16 (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
    return (uint32_t)__bfloat16_as_ushort(h2.x) | ((uint32_t)__bfloat16_as_ushort(h2.y) << 16);
}

template <bool OUT_NHWC, bool PAIRS>
__global__ void __launch_bounds__(256) stem_tc_bf16_kernel(const StemLaunch a, int n_mma, StemTcGeom g,
                                                           unsigned int *status) {
    constexpr int S = kStemTcStages;
    extern __shared__ uint8_t stem_smem_raw[];
    const uint32_t raw = ptx::smem_u32(stem_smem_raw);
    uint8_t *base = stem_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = base;                                           // S x 128 rows x 128 B
    uint8_t *sB = base + S * 16384;                               // 64 rows x 128 B
    float *sBias = reinterpret_cast<float *>(sB + 8192);          // 64
    uint64_t *bars = reinterpret_cast<uint64_t *>(sBias + 64);    // 2
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int row = t & 127, half = t >> 7;
    const int KK = a.KS * a.KS;
    const int kslices = PAIRS ? 3 : (KK + 3) / 4;    // 16-value K slices: 4 taps (or 2 pairs) each
    const uint32_t ncols = 2 * n_mma <= 32 ? 32u : (2 * n_mma <= 64 ? 64u : 128u);
    const bool silu = a.act != CBS_ACT_IDENTITY;
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), ncols);
        ptx::tmem_relinquish();
    }
    if (t == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
        ptx::fence_mbar_init();
    }
    // This CTA holds its tensor memory: the next grid may be scheduled.  Then
    // wait for the previous one before touching global memory.
    __syncthreads();
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    // B row co: the folded weights of output channel co in the K layout above,
    // zero for co >= C_out; 16-byte chunk q stored at q ^ (co % 8).
    const uint2 *w2 = static_cast<const uint2 *>(a.w);   // [C_out][KK] taps of 4 bf16
    for (int idx = t; idx < n_mma * 8; idx += 256) {
        const int co = idx >> 3, q = idx & 7;
        uint2 lo = make_uint2(0u, 0u), hi = make_uint2(0u, 0u);
        if (co < a.Cout) {
            const uint2 *wr = w2 + (size_t)co * KK;
            if (PAIRS) {
                if (q < 6) {
                    const int r = q >> 1;
                    if ((q & 1) == 0) {
                        hi = wr[r * 3];
                    } else {
                        lo = wr[r * 3 + 1];
                        hi = wr[r * 3 + 2];
                    }
                }
            } else {
                if (2 * q < KK) lo = wr[2 * q];
                if (2 * q + 1 < KK) hi = wr[2 * q + 1];
            }
        }
        *reinterpret_cast<uint4 *>(sB + co * 128 + ((q ^ (co & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    // Bias, halved for the tanh form of SiLU.
    if (t < 64) {
        const float b = t < a.Cout ? static_cast<const float *>(a.bias)[t] : 0.0f;
        sBias[t] = silu ? 0.5f * b : b;
    }

    const int n_local = (int)blockIdx.x < g.n_tiles ? (g.n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int ohw = a.OH * a.OW;
    const uint2 *x2 = static_cast<const uint2 *>(a.x);   // one 4-channel bf16 pixel
    const uint32_t sA_u32 = ptx::smem_u32(sA);
    const uint32_t swz = (uint32_t)(row & 7);

    // Issue this thread's copies of local tile i into stage i % S (an empty
    // group past the last tile).
    auto gather = [&](int i) {
        if (i < n_local) {
            const int pix = ((int)blockIdx.x + i * (int)gridDim.x) * 128 + row;
            const bool valid = pix < g.total;
            const int img = fast_div(pix, g.div_ohw);
            const int rem = pix - img * ohw;
            const int oh = fast_div(rem, g.div_ow);
            const int ow = rem - oh * a.OW;
            const uint32_t dst = sA_u32 + (uint32_t)((i % S) * 16384 + row * 128);
            if (PAIRS) {
#pragma unroll
                for (int qq = 0; qq < 3; ++qq) {
                    const int q = 3 * half + qq, r = q >> 1;
                    const int ih = 2 * oh - 1 + r, col = 2 * ow - 2 + 2 * (q & 1);
                    const bool in = valid && (unsigned)ih < (unsigned)a.H && col >= 0 && col + 1 < a.W;
                    const void *src = in ? (const void *)(x2 + (size_t)(img * a.H + ih) * a.W + col) : a.x;
                    ptx::cp_async_16(dst + (((uint32_t)q ^ swz) << 4), src, in ? 16u : 0u);
                }
            } else {
#pragma unroll
                for (int ss = 0; ss < 6; ++ss) {
                    const int s = 6 * half + ss;
                    if (s >= kslices * 4) break;
                    const int r = s / a.KS, c = s - (s / a.KS) * a.KS;
                    const int ih = oh * a.stride - a.pad + r, iw = ow * a.stride - a.pad + c;
                    const bool in = valid && s < KK && (unsigned)ih < (unsigned)a.H && (unsigned)iw < (unsigned)a.W;
                    const void *src = in ? (const void *)(x2 + (size_t)(img * a.H + ih) * a.W + iw) : a.x;
                    ptx::cp_async_8(dst + (((uint32_t)(s >> 1) ^ swz) << 4) + (uint32_t)((s & 1) * 8), src,
                                    in ? 8u : 0u);
                }
            }
        }
        ptx::cp_async_commit();
    };

    // Bias, activation, residual and stores of this thread's 8-channel groups
    // (half, half + 2, ...) of local tile i, from its accumulator.
    auto epilogue = [&](int i, uint32_t tmem) {
        const int pix = ((int)blockIdx.x + i * (int)gridDim.x) * 128 + row;
        const bool valid = pix < g.total;
        const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((i & 1) * n_mma);
        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(a.y);
        const __nv_bfloat16 *res = static_cast<const __nv_bfloat16 *>(a.residual);
        for (int c0 = 8 * half; c0 < n_mma; c0 += 16) {
            uint32_t v[8];
            ptx::tmem_ld8(t_row + (uint32_t)c0, v);
            ptx::tmem_ld_wait();
            if (!valid) continue;
            float o[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                o[jj] = silu ? silu_tanh(fmaf(__uint_as_float(v[jj]), 0.5f, sBias[c0 + jj]))
                             : __uint_as_float(v[jj]) + sBias[c0 + jj];
            if (OUT_NHWC && c0 + 8 <= a.Cout && (a.Cout & 7) == 0) {
                const size_t off = (size_t)pix * a.Cout + c0;
                if (res) {   // bf16 -> float is a 16-bit shift
                    const uint4 rv = *reinterpret_cast<const uint4 *>(res + off);
                    o[0] += __uint_as_float(rv.x << 16), o[1] += __uint_as_float(rv.x & 0xffff0000u);
                    o[2] += __uint_as_float(rv.y << 16), o[3] += __uint_as_float(rv.y & 0xffff0000u);
                    o[4] += __uint_as_float(rv.z << 16), o[5] += __uint_as_float(rv.z & 0xffff0000u);
                    o[6] += __uint_as_float(rv.w << 16), o[7] += __uint_as_float(rv.w & 0xffff0000u);
                }
                *reinterpret_cast<uint4 *>(y + off) = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                                                 pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
            } else {
                const int img = fast_div(pix, g.div_ohw);
                const int rem = pix - img * ohw;
                const int oh = fast_div(rem, g.div_ow);
                const int ow = rem - oh * a.OW;
                const size_t plane = (size_t)a.OH * a.out_row_stride;
                const size_t opix = (size_t)oh * a.out_row_stride + ow;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int c = c0 + jj;
                    if (c >= a.Cout) break;
                    const size_t off = OUT_NHWC ? (size_t)pix * a.Cout + c : ((size_t)img * a.Cout + c) * plane + opix;
                    const float r = res ? __bfloat162float(res[off]) : 0.0f;
                    y[off] = __float2bfloat16_rn(o[jj] + r);
                }
            }
        }
    };

#pragma unroll 1
    for (int i = 0; i < S - 1; ++i) gather(i);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t dhi = ptx::smem_desc(0u, 16u, 1024u, 2u);
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n_mma >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);
    const uint64_t bd = dhi | (uint64_t)((ptx::smem_u32(sB) & 0x3FFFFu) >> 4);
    bool failed = false;
#pragma unroll 1
    for (int i = 0; i <= n_local; ++i) {
        if (i < n_local) {
            ptx::cp_async_wait<S - 2>();   // this thread's copies of tile i have landed
            if (PAIRS) {                   // zero the unused first pixel of each pair this thread copied
                uint8_t *rp = sA + (i % S) * 16384 + row * 128;
                *reinterpret_cast<uint2 *>(rp + ((uint32_t)(half ? 4 : 0) ^ swz) * 16) = make_uint2(0u, 0u);
                if (!half) *reinterpret_cast<uint2 *>(rp + (2u ^ swz) * 16) = make_uint2(0u, 0u);
            }
            ptx::fence_proxy_async_smem();
        }
        ptx::tc_fence_before();
        if (__syncthreads_or(failed)) break;
        ptx::tc_fence_after();
        if (i < n_local && t == 0) {
            const uint64_t ad = dhi | (uint64_t)(((sA_u32 + (uint32_t)((i % S) * 16384)) & 0x3FFFFu) >> 4);
            const uint32_t acc = tmem + (uint32_t)((i & 1) * n_mma);
            for (int k = 0; k < kslices; ++k) ptx::mma_f16(acc, ad + 2u * k, bd + 2u * k, idesc, k > 0 ? 1u : 0u);
            ptx::mma_commit(ptx::smem_u32(&bars[i & 1]));
        }
        if (i > 0) {
            const int j = i - 1;
            bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&bars[j & 1]), (uint32_t)((j >> 1) & 1), kStemWaitNs);
            ok = __all_sync(0xffffffffu, ok);   // warp-uniform before .sync.aligned loads
            if (!ok) {
                failed = true;
                if (lane == 0) atomicOr(status, 1u);
            } else {
                ptx::tc_fence_after();
                epilogue(j, tmem);
            }
        }
        // Stage (i - 1) % S is free: its MMAs completed before the wait above.
        if (i < n_local) gather(i + S - 1);
    }
    ptx::cp_async_wait<0>();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

// The detector's BF16 and TF32 stems on a kernel of their own: 3x3, stride
// 2, pad 1 over 4-channel NHWC pixels of even input width W, 16 output
// channels, NHWC output, no residual.  The general kernel above gathers every output
// pixel's window from L2 (96 bytes per pixel, three times the input); this
// one walks whole output rows.  Each CTA takes a band of consecutive output
// rows (n, oh); one TMA box brings each input row into shared memory once
// (zero-filled above and below the image), and the CTA rewrites it as the
// rows of the MMA's A operand: for output column k, the pixel pair
// (2k-2, 2k-1) with its first pixel zeroed, then the pair (2k, 2k+1) (the
// pair K layout of the general kernel; the zeroed pixel's weights are zero,
// and zeroing it keeps a non-finite neighbour out of the sum): 32 bytes in
// BF16, stored 32-byte swizzled (one K=16 MMA per kernel row), 64 bytes in
// TF32, stored 64-byte swizzled (two K=8 MMAs).  Output row oh is, per kernel
// row r, ceil(OW / 128) M=128 tiles whose A is a 128-row slice of input row
// 2 oh - 1 + r's rewrite.  Input row 2 oh + 1 is also row 2 (oh + 1) - 1:
// each input row is loaded and rewritten once per band.
//
// Per step (one output row): warps 0-7 rewrite the step's new input rows
// (loaded kStemRowsAhead steps earlier); barrier; warp 8 issues the MMAs
// into accumulator buffer step % 2 and the input loads of step +
// kStemRowsAhead, while warps 0-7 wait for the previous step's MMAs and run
// its epilogue.  The issuing thread never waits on a barrier with its MMAs
// in flight (such a wait stalls it for ~700 cycles on GB300).  Rewrites go to a ring of kStemRowsESlots slots: step s writes
// slots 2s, 2s+1 (mod 6) and its MMAs read 2s-1 .. 2s+1, so a slot is
// rewritten only after the MMAs of steps s-2 and s-3 -- both waited for --
// have read it.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

struct StemRowsGeom {
    int rows;        // output rows N * OH
    int mtiles;      // M=128 tiles per output row: ceil(OW / 128)
    int eslot;       // bytes of one rewritten input row: mtiles * 128 * (A row bytes)
    int raw;         // bytes of one input row: W * (pixel bytes)
    int rawstride;   // bytes between raw row slots: raw rounded up to 1024 (B stays swizzle-aligned)
    FastDiv div_oh;  // by OH: output row R = img * OH + oh
};

// Offset of 16-byte chunk c of A row k in a slot of ER-byte rows, swizzled
// as TMA and the tensor cores swizzle them (16-byte chunk bits XOR address
// bits 7.. : one bit for 32-byte rows, two for 64-byte rows).
template <int ER>
__device__ __forceinline__ uint32_t rows_chunk(int k, int c) {
    return ER == 32 ? (uint32_t)(k * 32 + ((c ^ ((k >> 2) & 1)) << 4))
                    : (uint32_t)(k * 64 + ((c ^ ((k >> 1) & 3)) << 4));
}

// KIND 1: BF16 pixels (8 bytes); KIND 3: TF32, float pixels (16 bytes).
template <int KIND, bool SILU>
__global__ void __launch_bounds__(kStemRowsThreads) stem_tc_rows_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                        const StemLaunch a, StemRowsGeom g,
                                                                        unsigned int *status) {
    constexpr int D = kStemRowsAhead, NE = kStemRowsESlots;
    constexpr int PX = KIND == 3 ? 16 : 8;     // bytes of one input pixel
    constexpr int ER = 4 * PX;                 // bytes of one A row (one kernel row of one output column)
    constexpr int TILE = 128 * ER;             // bytes of one M=128 slice of a rewritten row
    constexpr int NW = kStemRowsThreads / 32 - 1;   // rewrite and epilogue warps; warp NW issues
    extern __shared__ uint8_t stem_smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(stem_smem_raw);
    uint8_t *base = stem_smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    uint8_t *sE = base;                                           // NE rewritten rows
    uint8_t *sR = sE + NE * g.eslot;                              // 2D + 1 raw input rows
    uint8_t *sB = sR + (2 * D + 1) * g.rawstride;                 // 3 kernel rows x 16 x ER bytes
    float *sBias = reinterpret_cast<float *>(sB + 3 * 16 * ER);   // 16, halved (tanh form of SiLU)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sBias + 16);    // raw_full[D], mma_done[2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + D + 2);
    const uint32_t sE_u32 = ptx::smem_u32(sE), sR_u32 = ptx::smem_u32(sR), sB_u32 = ptx::smem_u32(sB);
    auto raw_bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    auto mma_bar = [&](int i) { return ptx::smem_u32(&bars[D + i]); };

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const uint32_t tcols = 2 * g.mtiles * 16 <= 32 ? 32u : (2 * g.mtiles * 16 <= 64 ? 64u : 128u);
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), tcols);   // two buffers x mtiles x 16 columns
        ptx::tmem_relinquish();
    }
    if (t == 0) {
        for (int i = 0; i < D + 2; ++i) ptx::mbar_init(ptx::smem_u32(&bars[i]), 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmX);
    }
    __syncthreads();
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    // B for kernel row r at sB + 16 ER r: output channel co's ER bytes in the
    // A rows' layout: (0, tap (r, 0)), then (tap (r, 1), tap (r, 2)).
    if (t < 48) {
        const int r = t >> 4, co = t & 15;
        uint8_t *rowp = sB + r * 16 * ER;
        if (KIND == 1) {
            const uint2 *wr = static_cast<const uint2 *>(a.w) + co * 9 + 3 * r;   // [16][9] taps of 4 bf16
            const uint2 w0 = wr[0], w1 = wr[1], w2 = wr[2];
            *reinterpret_cast<uint4 *>(rowp + rows_chunk<ER>(co, 0)) = make_uint4(0u, 0u, w0.x, w0.y);
            *reinterpret_cast<uint4 *>(rowp + rows_chunk<ER>(co, 1)) = make_uint4(w1.x, w1.y, w2.x, w2.y);
        } else {
            const uint4 *wr = static_cast<const uint4 *>(a.w) + co * 9 + 3 * r;   // [16][9] taps of 4 floats
            *reinterpret_cast<uint4 *>(rowp + rows_chunk<ER>(co, 0)) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int c = 0; c < 3; ++c) *reinterpret_cast<uint4 *>(rowp + rows_chunk<ER>(co, c + 1)) = wr[c];
        }
    }
    if (t < 16) sBias[t] = 0.5f * static_cast<const float *>(a.bias)[t];

    // This CTA's band of output rows.
    const int R0 = (int)((long long)blockIdx.x * g.rows / gridDim.x);
    const int nsteps = (int)((long long)(blockIdx.x + 1) * g.rows / gridDim.x) - R0;
    const int OW = a.OW;
    // Input loads of step s (one TMA box per input row), issued by lanes 0-2
    // of the calling warp in parallel (a thread waits ~570 cycles per box):
    // rows 2 oh and 2 oh + 1 into raw slots 2s, 2s + 1 (mod 2D), and at the
    // band's first step row 2 oh - 1 into slot 2D.
    auto issue_loads = [&](int s) {
        const int R = R0 + s, img = fast_div(R, g.div_oh), oh = R - img * a.OH;
        const bool with_a = s == 0 && oh > 0;
        const uint32_t bar = raw_bar(s % D);
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar, (uint32_t)((with_a ? 3 : 2) * g.raw));
        __syncwarp();
        if (lane < 2)
            ptx::tma_load_4d(sR_u32 + (uint32_t)(((2 * s + lane) % (2 * D)) * g.rawstride), &tmX, bar, 0, 0,
                             2 * oh + lane, img);
        else if (lane == 2 && with_a)
            ptx::tma_load_4d(sR_u32 + (uint32_t)(2 * D * g.rawstride), &tmX, bar, 0, 0, 2 * oh - 1, img);
    };
    // Rewrite raw slot `rs` into A-row slot `es` (column k: pair k-1 with its
    // first pixel zeroed, then pair k).
    auto rewrite = [&](int rs, int es) {
        const uint8_t *rp = sR + rs * g.rawstride;
        uint8_t *ep = sE + es * g.eslot;
        for (int k = t; k < OW; k += 32 * NW) {   // warps 0 .. NW-1
            if (KIND == 1) {
                const uint4 pk = *reinterpret_cast<const uint4 *>(rp + 16 * k);
                const uint2 pm = k > 0 ? *reinterpret_cast<const uint2 *>(rp + 16 * k - 8) : make_uint2(0u, 0u);
                *reinterpret_cast<uint4 *>(ep + rows_chunk<ER>(k, 0)) = make_uint4(0u, 0u, pm.x, pm.y);
                *reinterpret_cast<uint4 *>(ep + rows_chunk<ER>(k, 1)) = pk;
            } else {
                const uint4 pm = k > 0 ? *reinterpret_cast<const uint4 *>(rp + 32 * k - 16) : make_uint4(0u, 0u, 0u, 0u);
                const uint4 p0 = *reinterpret_cast<const uint4 *>(rp + 32 * k);
                const uint4 p1 = *reinterpret_cast<const uint4 *>(rp + 32 * k + 16);
                *reinterpret_cast<uint4 *>(ep + rows_chunk<ER>(k, 0)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(ep + rows_chunk<ER>(k, 1)) = pm;
                *reinterpret_cast<uint4 *>(ep + rows_chunk<ER>(k, 2)) = p0;
                *reinterpret_cast<uint4 *>(ep + rows_chunk<ER>(k, 3)) = p1;
            }
        }
    };

    if (warp == NW)
        for (int s = 0; s < D && s < nsteps; ++s) issue_loads(s);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    float bh[8];
    const int q = warp & 3, h = (warp >> 2) & 1;   // TMEM lane quadrant, column half (8 h .. 8 h + 7)
#pragma unroll
    for (int c = 0; c < 8; ++c) bh[c] = sBias[8 * h + c];
    // ER-byte rows, 8-row groups 8 ER apart; swizzle code 6 (32 B) or 4 (64 B).
    const uint64_t dsw = ptx::smem_desc(0u, 16u, 8u * ER, ER == 32 ? 6u : 4u);
    constexpr uint32_t fmt = KIND == 3 ? 2u : 1u;   // TF32 : BF16 operands
    const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(16 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const int bufcols = g.mtiles * 16;
    bool failed = false;
    const bool issuer = warp == NW;
    int issued = D < nsteps ? D : nsteps;   // steps whose loads have been issued (thread 0, then warp 8)
    int stop = nsteps;                      // loads of steps >= stop may still be in flight at exit
#pragma unroll 1
    for (int s = 0; s <= nsteps; ++s) {
        if (s < nsteps && !issuer) {
            if (!ptx::mbar_wait_bounded(raw_bar(s % D), (uint32_t)((s / D) & 1), kStemWaitNs)) {
                failed = true;
                if (lane == 0) atomicOr(status, 1u);
            } else {
                const int R = R0 + s, oh = R - fast_div(R, g.div_oh) * a.OH;
                rewrite((2 * s) % (2 * D), (2 * s) % NE);
                rewrite((2 * s + 1) % (2 * D), (2 * s + 1) % NE);
                if (s == 0 && oh > 0) rewrite(2 * D, NE - 1);
                ptx::fence_proxy_async_smem();
            }
        }
        ptx::tc_fence_before();
        if (__syncthreads_or(failed)) {
            stop = s;
            break;
        }
        ptx::tc_fence_after();
        if (issuer) {
            if (s >= nsteps) continue;
            const int R = R0 + s, oh = R - fast_div(R, g.div_oh) * a.OH;
            if (lane == 0) {
                const int r0 = oh == 0 ? 1 : 0;   // kernel row 0 of output row 0 is padding
                const uint32_t d0 = tmem + (uint32_t)((s & 1) * bufcols);
                for (int r = r0; r < 3; ++r) {
                    const int es = ((2 * s - 1 + r) % NE + NE) % NE;
                    const uint64_t bd = dsw | (uint64_t)(((sB_u32 + (uint32_t)(r * 16 * ER)) & 0x3FFFFu) >> 4);
                    for (int m = 0; m < g.mtiles; ++m) {
                        const uint64_t ad =
                            dsw | (uint64_t)(((sE_u32 + (uint32_t)(es * g.eslot + m * TILE)) & 0x3FFFFu) >> 4);
                        if (KIND == 1) {
                            ptx::mma_f16(d0 + (uint32_t)(m * 16), ad, bd, idesc, r > r0 ? 1u : 0u);
                        } else {   // two K=8 slices, 32 bytes apart
                            ptx::mma_tf32(d0 + (uint32_t)(m * 16), ad, bd, idesc, r > r0 ? 1u : 0u);
                            ptx::mma_tf32(d0 + (uint32_t)(m * 16), ad + 2u, bd + 2u, idesc, 1u);
                        }
                    }
                }
                ptx::mma_commit(mma_bar(s & 1));
            }
            // Step s's raw slots and load barrier are free: they take step s + D.
            if (s + D < nsteps) {
                issue_loads(s + D);
                issued = s + D + 1;
            }
            continue;
        }
        if (s == 0) continue;
        const int j = s - 1;
        bool ok = ptx::mbar_wait_bounded(mma_bar(j & 1), (uint32_t)((j >> 1) & 1), kStemWaitNs);
        ok = __all_sync(0xffffffffu, ok);   // warp-uniform before .sync.aligned loads
        if (!ok) {
            failed = true;
            if (lane == 0) atomicOr(status, 1u);
            continue;
        }
        ptx::tc_fence_after();
        // Epilogue of output row R0 + j: this warp's 32 TMEM lanes of each
        // M tile, output channels 8 h .. 8 h + 7.
        const size_t pix0 = (size_t)(R0 + j) * OW;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((j & 1) * bufcols + 8 * h);
        uint32_t v[kStemRowsMaxMtiles][8];
#pragma unroll
        for (int m = 0; m < kStemRowsMaxMtiles; ++m)
            if (m < g.mtiles && m * 128 + 32 * q < OW) ptx::tmem_ld8(tl + (uint32_t)(m * 16), v[m]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < kStemRowsMaxMtiles; ++m) {
            const int k = m * 128 + 32 * q + lane;
            if (m < g.mtiles && k < OW) {
                float o[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float hv = fmaf(__uint_as_float(v[m][c]), 0.5f, bh[c]);
                    o[c] = SILU ? silu_tanh(hv) : hv + hv;
                }
                const size_t off = (pix0 + (size_t)k) * 16 + 8 * h;
                if (KIND == 1) {
                    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.y) + off) =
                        make_uint4(cvt_bf16x2(o[0], o[1]), cvt_bf16x2(o[2], o[3]), cvt_bf16x2(o[4], o[5]),
                                   cvt_bf16x2(o[6], o[7]));
                } else {
                    float4 *yp = reinterpret_cast<float4 *>(static_cast<float *>(a.y) + off);
                    yp[0] = make_float4(o[0], o[1], o[2], o[3]);
                    yp[1] = make_float4(o[4], o[5], o[6], o[7]);
                }
            }
        }
    }
    // After a timeout: let the loads already issued land before the CTA exits.
    if (issuer && lane == 0)
        for (int k = stop; k < issued; ++k)
            ptx::mbar_wait_bounded(raw_bar(k % D), (uint32_t)((k / D) & 1), kStemWaitNs);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, tcols);
    }
}

// INT8 codes widened to bfloat16 (exact for |q| <= 128: the float has at most
// 8 significant bits, so its top 16 bits are the bfloat16).
__device__ __forceinline__ uint32_t codes_to_bf16x2(int lo, int hi) {
    return (__float_as_uint((float)lo) >> 16) | (__float_as_uint((float)hi) & 0xffff0000u);
}

// Four int8 codes (one pixel, 4 channels) -> four bfloat16.
__device__ __forceinline__ uint2 pixel_codes_to_bf16(uint32_t w) {
    const int c0 = (int)(w << 24) >> 24, c1 = (int)(w << 16) >> 24, c2 = (int)(w << 8) >> 24, c3 = (int)w >> 24;
    return make_uint2(codes_to_bf16x2(c0, c1), codes_to_bf16x2(c2, c3));
}

// INT8 stem on the tensor cores: the BF16 kernel's layout and pipeline, with
// the gather through registers (codes are widened to bfloat16 on their way
// into the A tile, one tile ahead of the MMA; a tap outside the image reads
// the code of zero, z_x) and the specified requantising epilogue.  The sums
// are exact: at most 48 products of magnitude <= 16256 per output.
template <bool OUT_NHWC, bool PAIRS>
__global__ void __launch_bounds__(256) stem_tc_i8_kernel(const StemLaunch a, int n_mma, StemTcGeom g,
                                                         unsigned int *status) {
    static_assert(kStemTcStages >= 2, "the INT8 stem uses two A stages");
    extern __shared__ uint8_t stem_smem_raw[];
    const uint32_t raw = ptx::smem_u32(stem_smem_raw);
    uint8_t *base = stem_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = base;                                           // 2 x 128 rows x 128 B
    uint8_t *sB = base + kStemTcStages * 16384;                   // 64 rows x 128 B
    int32_t *sBias = reinterpret_cast<int32_t *>(sB + 8192);      // 64: int32 bias (with the zero point)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sBias + 64);    // 2
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
    __shared__ float sMc[64];

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int row = t & 127, half = t >> 7;
    const int KK = a.KS * a.KS;
    const int kslices = PAIRS ? 3 : (KK + 3) / 4;
    const uint32_t ncols = 2 * n_mma <= 32 ? 32u : (2 * n_mma <= 64 ? 64u : 128u);
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), ncols);
        ptx::tmem_relinquish();
    }
    if (t == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::griddep_launch_dependents();   // after this CTA's TMEM allocation
    ptx::griddep_wait();
    // B: the weight codes (bf16) in the BF16 stem's K layout.
    const uint2 *w2 = static_cast<const uint2 *>(a.w);
    for (int idx = t; idx < n_mma * 8; idx += 256) {
        const int co = idx >> 3, q = idx & 7;
        uint2 lo = make_uint2(0u, 0u), hi = make_uint2(0u, 0u);
        if (co < a.Cout) {
            const uint2 *wr = w2 + (size_t)co * KK;
            if (PAIRS) {
                if (q < 6) {
                    const int r = q >> 1;
                    if ((q & 1) == 0) {
                        hi = wr[r * 3];
                    } else {
                        lo = wr[r * 3 + 1];
                        hi = wr[r * 3 + 2];
                    }
                }
            } else {
                if (2 * q < KK) lo = wr[2 * q];
                if (2 * q + 1 < KK) hi = wr[2 * q + 1];
            }
        }
        *reinterpret_cast<uint4 *>(sB + co * 128 + ((q ^ (co & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    if (t < 64) {
        sBias[t] = t < a.Cout ? static_cast<const int32_t *>(a.bias)[t] : 0;
        sMc[t] = t < a.Cout ? a.m_c[t] : 0.0f;
    }

    const int n_local = (int)blockIdx.x < g.n_tiles ? (g.n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int ohw = a.OH * a.OW;
    const uint32_t *x4 = static_cast<const uint32_t *>(a.x);   // one 4-channel int8 pixel
    const uint32_t zfill = (uint32_t)(uint8_t)(int8_t)a.zp_x * 0x01010101u;
    const uint32_t swz = (uint32_t)(row & 7);

    // This thread's share of one tile's taps, as raw codes (PAIRS: three
    // 2-pixel chunks; otherwise six single taps).
    uint32_t reg[6];
    auto load = [&](int i) {
        const int pix = ((int)blockIdx.x + i * (int)gridDim.x) * 128 + row;
        const bool valid = pix < g.total;
        const int img = fast_div(pix, g.div_ohw);
        const int rem = pix - img * ohw;
        const int oh = fast_div(rem, g.div_ow);
        const int ow = rem - oh * a.OW;
        if (PAIRS) {
#pragma unroll
            for (int qq = 0; qq < 3; ++qq) {
                const int q = 3 * half + qq, r = q >> 1;
                const int ih = 2 * oh - 1 + r, col = 2 * ow - 2 + 2 * (q & 1);
                const bool in = valid && (unsigned)ih < (unsigned)a.H && col >= 0 && col + 1 < a.W;
                uint2 v = make_uint2(zfill, zfill);
                if (in) v = __ldg(reinterpret_cast<const uint2 *>(x4 + (size_t)(img * a.H + ih) * a.W + col));
                reg[2 * qq] = v.x;
                reg[2 * qq + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int ss = 0; ss < 6; ++ss) {
                const int s2 = 6 * half + ss;
                const int r = s2 / a.KS, c = s2 - (s2 / a.KS) * a.KS;
                const int ih = oh * a.stride - a.pad + r, iw = ow * a.stride - a.pad + c;
                const bool in = valid && s2 < KK && (unsigned)ih < (unsigned)a.H && (unsigned)iw < (unsigned)a.W;
                reg[ss] = in ? __ldg(x4 + (size_t)(img * a.H + ih) * a.W + iw) : zfill;
            }
        }
    };
    // Widen the loaded codes into stage st of A.
    auto store = [&](int st) {
        uint8_t *rp = sA + st * 16384 + row * 128;
        if (PAIRS) {
#pragma unroll
            for (int qq = 0; qq < 3; ++qq) {
                const int q = 3 * half + qq;
                const uint2 lo = pixel_codes_to_bf16(reg[2 * qq]), hi = pixel_codes_to_bf16(reg[2 * qq + 1]);
                *reinterpret_cast<uint4 *>(rp + (((uint32_t)q ^ swz) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
        } else {
#pragma unroll
            for (int ss = 0; ss < 6; ++ss) {
                const int s2 = 6 * half + ss;
                if (s2 >= kslices * 4) break;
                *reinterpret_cast<uint2 *>(rp + (((uint32_t)(s2 >> 1) ^ swz) << 4) + (s2 & 1) * 8) =
                    pixel_codes_to_bf16(reg[ss]);
            }
        }
    };
    // Requantising epilogue of this thread's 8-channel groups of local tile i.
    auto epilogue = [&](int i, uint32_t tmem) {
        const int pix = ((int)blockIdx.x + i * (int)gridDim.x) * 128 + row;
        const bool valid = pix < g.total;
        const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((i & 1) * n_mma);
        int8_t *y = static_cast<int8_t *>(a.y);
        for (int c0 = 8 * half; c0 < n_mma; c0 += 16) {
            uint32_t v[8];
            ptx::tmem_ld8(t_row + (uint32_t)c0, v);
            ptx::tmem_ld_wait();
            if (!valid) continue;
            int q[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int acc = (int)((unsigned)__float2int_rn(__uint_as_float(v[jj])) + (unsigned)sBias[c0 + jj]);
                q[jj] = requant_i8_fast(acc, sMc[c0 + jj], a.inv_s_y, a.zp_y);
            }
            if (OUT_NHWC && c0 + 8 <= a.Cout && (a.Cout & 7) == 0) {
                uint32_t lo = 0u, hi = 0u;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    lo |= (uint32_t)(uint8_t)(int8_t)q[jj] << (8 * jj);
                    hi |= (uint32_t)(uint8_t)(int8_t)q[jj + 4] << (8 * jj);
                }
                *reinterpret_cast<uint2 *>(y + (size_t)pix * a.Cout + c0) = make_uint2(lo, hi);
            } else {
                const int img = fast_div(pix, g.div_ohw);
                const int rem = pix - img * ohw;
                const int oh = fast_div(rem, g.div_ow);
                const int ow = rem - oh * a.OW;
                const size_t plane = (size_t)a.OH * a.out_row_stride;
                const size_t opix = (size_t)oh * a.out_row_stride + ow;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int c = c0 + jj;
                    if (c >= a.Cout) break;
                    const size_t off = OUT_NHWC ? (size_t)pix * a.Cout + c : ((size_t)img * a.Cout + c) * plane + opix;
                    y[off] = (int8_t)q[jj];
                }
            }
        }
    };

    if (n_local > 0) {
        load(0);
        store(0);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t dhi = ptx::smem_desc(0u, 16u, 1024u, 2u);
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n_mma >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);
    const uint64_t bd = dhi | (uint64_t)((ptx::smem_u32(sB) & 0x3FFFFu) >> 4);
    const uint32_t sA_u32 = ptx::smem_u32(sA);
    bool failed = false;
#pragma unroll 1
    for (int i = 0; i <= n_local; ++i) {
        if (i + 1 < n_local) load(i + 1);   // in flight during this tile's MMA and the last tile's epilogue
        ptx::fence_proxy_async_smem();       // stage i % 2 written through the generic proxy
        ptx::tc_fence_before();
        if (__syncthreads_or(failed)) break;
        ptx::tc_fence_after();
        if (i < n_local && t == 0) {
            const uint64_t ad = dhi | (uint64_t)(((sA_u32 + (uint32_t)((i & 1) * 16384)) & 0x3FFFFu) >> 4);
            const uint32_t acc = tmem + (uint32_t)((i & 1) * n_mma);
            for (int k = 0; k < kslices; ++k) ptx::mma_f16(acc, ad + 2u * k, bd + 2u * k, idesc, k > 0 ? 1u : 0u);
            ptx::mma_commit(ptx::smem_u32(&bars[i & 1]));
        }
        if (i > 0) {
            const int j = i - 1;
            bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&bars[j & 1]), (uint32_t)((j >> 1) & 1), kStemWaitNs);
            ok = __all_sync(0xffffffffu, ok);   // warp-uniform before .sync.aligned loads
            if (!ok) {
                failed = true;
                if (lane == 0) atomicOr(status, 1u);
            } else {
                ptx::tc_fence_after();
                epilogue(j, tmem);
            }
        }
        // Stage (i + 1) % 2 was read by the MMAs of tile i - 1, complete above.
        if (i + 1 < n_local && !failed) store((i + 1) & 1);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

// TF32 stem on the tensor cores.  An fp32 pixel of 4 channels is 16 bytes,
// so each tap is one 16-byte cp.async straight into the A tile (no
// conversion), and a tcgen05 kind::tf32 K slice (8 values, 32 bytes) holds two
// taps.  Nine taps (+ one zero slot) are five K slices, each its own
// 32-byte-swizzled block (128 rows x 32 B for A, 64 rows x 32 B for B), so no
// byte of shared memory is padding: 20 KB per A stage, two stages, four CTAs
// per SM.  Otherwise the BF16 kernel's pipeline (ring one tile ahead,
// double-buffered accumulators).
template <bool OUT_NHWC>
__global__ void __launch_bounds__(256) stem_tc_tf32_kernel(const StemLaunch a, int n_mma, StemTcGeom g,
                                                           unsigned int *status) {
    constexpr int S = 2, kSliceA = 4096, kSliceB = 2048, kStage = 5 * kSliceA;
    extern __shared__ uint8_t stem_smem_raw[];
    const uint32_t raw = ptx::smem_u32(stem_smem_raw);
    uint8_t *base = stem_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = base;                                             // S stages x 5 slices x 128 rows x 32 B
    uint8_t *sB = base + S * kStage;                                // 5 slices x 64 rows x 32 B
    float *sBias = reinterpret_cast<float *>(sB + 5 * kSliceB);     // 64
    uint64_t *bars = reinterpret_cast<uint64_t *>(sBias + 64);      // 2
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int row = t & 127, half = t >> 7;
    const int KK = a.KS * a.KS;
    const int kslices = (KK + 1) / 2;                 // two taps per K slice
    const uint32_t ncols = 2 * n_mma <= 32 ? 32u : (2 * n_mma <= 64 ? 64u : 128u);
    const bool silu = a.act != CBS_ACT_IDENTITY;
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), ncols);
        ptx::tmem_relinquish();
    }
    if (t == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::griddep_launch_dependents();   // after this CTA's TMEM allocation
    ptx::griddep_wait();
    // B row co, slot s: tap s's four folded weights (zero past KK and for
    // co >= C_out), slice s / 2, 16-byte chunk s % 2 stored at (s % 2) ^ bit 2 of co.
    const float4 *w4 = static_cast<const float4 *>(a.w);   // [C_out][KK] taps of 4 floats
    for (int idx = t; idx < n_mma * 10; idx += 256) {
        const int co = idx / 10, sl = idx - co * 10;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (co < a.Cout && sl < KK) v = w4[(size_t)co * KK + sl];
        *reinterpret_cast<float4 *>(sB + (sl >> 1) * kSliceB + co * 32 + (((sl & 1) ^ ((co >> 2) & 1)) << 4)) = v;
    }
    if (t < 64) {   // halved for the tanh form of SiLU
        const float b = t < a.Cout ? static_cast<const float *>(a.bias)[t] : 0.0f;
        sBias[t] = silu ? 0.5f * b : b;
    }

    const int n_local = (int)blockIdx.x < g.n_tiles ? (g.n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int ohw = a.OH * a.OW;
    const float4 *x4 = static_cast<const float4 *>(a.x);   // one 4-channel fp32 pixel
    const uint32_t sA_u32 = ptx::smem_u32(sA);
    const uint32_t swz = (uint32_t)((row >> 2) & 1);

    // This thread's five tap slots (5 * half ..) of local tile i into stage i % 2.
    auto gather = [&](int i) {
        if (i < n_local) {
            const int pix = ((int)blockIdx.x + i * (int)gridDim.x) * 128 + row;
            const bool valid = pix < g.total;
            const int img = fast_div(pix, g.div_ohw);
            const int rem = pix - img * ohw;
            const int oh = fast_div(rem, g.div_ow);
            const int ow = rem - oh * a.OW;
            const uint32_t dst = sA_u32 + (uint32_t)((i & 1) * kStage + row * 32);
#pragma unroll
            for (int ss = 0; ss < 5; ++ss) {
                const int sl = 5 * half + ss;
                if (sl >= 2 * kslices) break;
                const int r = sl / a.KS, c = sl - (sl / a.KS) * a.KS;
                const int ih = oh * a.stride - a.pad + r, iw = ow * a.stride - a.pad + c;
                const bool in = valid && sl < KK && (unsigned)ih < (unsigned)a.H && (unsigned)iw < (unsigned)a.W;
                const void *src = in ? (const void *)(x4 + (size_t)(img * a.H + ih) * a.W + iw) : a.x;
                ptx::cp_async_16(dst + (uint32_t)((sl >> 1) * kSliceA) + (((uint32_t)(sl & 1) ^ swz) << 4), src,
                                 in ? 16u : 0u);
            }
        }
        ptx::cp_async_commit();
    };

    // Bias, activation, residual and float stores of this thread's 8-channel
    // groups (half, half + 2, ...) of local tile i.
    auto epilogue = [&](int i, uint32_t tmem) {
        const int pix = ((int)blockIdx.x + i * (int)gridDim.x) * 128 + row;
        const bool valid = pix < g.total;
        const uint32_t t_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((i & 1) * n_mma);
        float *y = static_cast<float *>(a.y);
        const float *res = static_cast<const float *>(a.residual);
        for (int c0 = 8 * half; c0 < n_mma; c0 += 16) {
            uint32_t v[8];
            ptx::tmem_ld8(t_row + (uint32_t)c0, v);
            ptx::tmem_ld_wait();
            if (!valid) continue;
            float o[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                o[jj] = silu ? silu_tanh(fmaf(__uint_as_float(v[jj]), 0.5f, sBias[c0 + jj]))
                             : __uint_as_float(v[jj]) + sBias[c0 + jj];
            if (OUT_NHWC && c0 + 8 <= a.Cout && (a.Cout & 3) == 0) {
                const size_t off = (size_t)pix * a.Cout + c0;
                if (res) {
                    const float4 r0 = *reinterpret_cast<const float4 *>(res + off);
                    const float4 r1 = *reinterpret_cast<const float4 *>(res + off + 4);
                    o[0] += r0.x, o[1] += r0.y, o[2] += r0.z, o[3] += r0.w;
                    o[4] += r1.x, o[5] += r1.y, o[6] += r1.z, o[7] += r1.w;
                }
                *reinterpret_cast<float4 *>(y + off) = make_float4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<float4 *>(y + off + 4) = make_float4(o[4], o[5], o[6], o[7]);
            } else {
                const int img = fast_div(pix, g.div_ohw);
                const int rem = pix - img * ohw;
                const int oh = fast_div(rem, g.div_ow);
                const int ow = rem - oh * a.OW;
                const size_t plane = (size_t)a.OH * a.out_row_stride;
                const size_t opix = (size_t)oh * a.out_row_stride + ow;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int c = c0 + jj;
                    if (c >= a.Cout) break;
                    const size_t off = OUT_NHWC ? (size_t)pix * a.Cout + c : ((size_t)img * a.Cout + c) * plane + opix;
                    y[off] = o[jj] + (res ? res[off] : 0.0f);
                }
            }
        }
    };

    gather(0);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t dhi = ptx::smem_desc(0u, 16u, 256u, 6u);   // 32-byte swizzle, 8-row groups 256 B apart
    const uint32_t idesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n_mma >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);
    const uint32_t sB_u32 = ptx::smem_u32(sB);
    bool failed = false;
#pragma unroll 1
    for (int i = 0; i <= n_local; ++i) {
        if (i < n_local) {
            ptx::cp_async_wait<0>();   // this thread's copies of tile i have landed
            ptx::fence_proxy_async_smem();
        }
        ptx::tc_fence_before();
        if (__syncthreads_or(failed)) break;
        ptx::tc_fence_after();
        if (i < n_local && t == 0) {
            const uint32_t stage = sA_u32 + (uint32_t)((i & 1) * kStage);
            const uint32_t acc = tmem + (uint32_t)((i & 1) * n_mma);
            for (int k = 0; k < kslices; ++k) {
                const uint64_t ad = dhi | (uint64_t)(((stage + (uint32_t)(k * kSliceA)) & 0x3FFFFu) >> 4);
                const uint64_t bd = dhi | (uint64_t)(((sB_u32 + (uint32_t)(k * kSliceB)) & 0x3FFFFu) >> 4);
                ptx::mma_tf32(acc, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
            ptx::mma_commit(ptx::smem_u32(&bars[i & 1]));
        }
        if (i > 0) {
            const int j = i - 1;
            bool ok = ptx::mbar_wait_bounded(ptx::smem_u32(&bars[j & 1]), (uint32_t)((j >> 1) & 1), kStemWaitNs);
            ok = __all_sync(0xffffffffu, ok);   // warp-uniform before .sync.aligned loads
            if (!ok) {
                failed = true;
                if (lane == 0) atomicOr(status, 1u);
            } else {
                ptx::tc_fence_after();
                epilogue(j, tmem);
            }
        }
        // Stage (i + 1) % 2 was read by the MMAs of tile i - 1, complete above.
        if (i < n_local) gather(i + 1);
    }
    ptx::cp_async_wait<0>();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

}  // namespace

bool stem_uses_tensor_cores(int kind, int in_nhwc, int c_pad, int ks, int cout, long long pixels) {
    return (kind == 1 || kind == 2 || kind == 3) && in_nhwc && c_pad == 4 && ks <= 3 && cout <= 64 &&
           pixels < kStemTcMaxPixels;
}

namespace {

template <bool OUT_NHWC, bool PAIRS>
cudaError_t launch_stem_tc_as(const StemLaunch &L, int n_mma, StemTcGeom g, int grid, cudaStream_t s,
                              unsigned int *status) {
    auto kern = L.kind == 2 ? stem_tc_i8_kernel<OUT_NHWC, PAIRS> : stem_tc_bf16_kernel<OUT_NHWC, PAIRS>;
    const cudaError_t e = set_max_dyn_smem(kern, kStemTcSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, 256, kStemTcSmemBytes, s, L, n_mma, g, status);
}

template <bool OUT_NHWC>
cudaError_t launch_stem_tf32(const StemLaunch &L, int n_mma, StemTcGeom g, int grid, cudaStream_t s,
                             unsigned int *status) {
    auto kern = stem_tc_tf32_kernel<OUT_NHWC>;
    const cudaError_t e = set_max_dyn_smem(kern, kStemTf32SmemBytes);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, 256, kStemTf32SmemBytes, s, L, n_mma, g, status);
}

cudaError_t launch_stem_tc(const StemLaunch &L, cudaStream_t s) {
    unsigned int *status = device_status_word();
    if (!status) return cudaErrorInvalidValue;
    const long long total = (long long)L.N * L.OH * L.OW;
    if (total >= kStemTcMaxPixels) return cudaErrorInvalidValue;
    StemTcGeom g;
    g.total = (int)total;
    g.n_tiles = (int)((total + 127) / 128);
    g.div_ohw = make_fastdiv((uint32_t)(L.OH * L.OW));
    g.div_ow = make_fastdiv((uint32_t)L.OW);
    const int rk = L.tf32 ? 3 : L.kind;   // the row kernel's kind: 1 BF16, 3 TF32
    if (stem_s2_kernel_applies(rk, L.KS, L.stride, L.pad, L.W, L.Cout, L.out_nhwc, L.residual != nullptr)) {
        // Input rows as [N][H][nb][bx] elements (bx: the largest multiple of
        // 16 bytes dividing a row, at most 256 elements): one TMA box
        // {bx, nb, 1, 1} per row.
        const int esz = rk == 3 ? 4 : 2, px = 4 * esz;
        const int row_el = 4 * L.W, unit = 16 / esz;
        int bx = 0;
        for (int c = unit; c <= 256 && c <= row_el; c += unit)
            if (row_el % c == 0) bx = c;
        if (bx == 0) return cudaErrorInvalidValue;
        const int nb = row_el / bx;
        if (nb > 256) return cudaErrorInvalidValue;
        const cuuint64_t dims[4] = {(cuuint64_t)bx, (cuuint64_t)nb, (cuuint64_t)L.H, (cuuint64_t)L.N};
        const cuuint64_t strides[3] = {(cuuint64_t)bx * esz, (cuuint64_t)L.W * px, (cuuint64_t)L.H * L.W * px};
        const cuuint32_t box[4] = {(cuuint32_t)bx, (cuuint32_t)nb, 1u, 1u};
        CUtensorMap tm;
        if (encode_plain_map(&tm, rk == 3 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, L.x,
                             dims, strides, box) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        StemRowsGeom rg;
        rg.rows = L.N * L.OH;
        rg.mtiles = (L.OW + 127) / 128;
        rg.eslot = rg.mtiles * 128 * 4 * px;
        rg.raw = L.W * px;
        rg.rawstride = (rg.raw + 1023) / 1024 * 1024;
        rg.div_oh = make_fastdiv((uint32_t)L.OH);
        const int smem = stem_rows_smem_bytes(rk, L.W);
        const int grid = std::min(rg.rows, L.grid);   // the plan's CTAs, one band of output rows each
        const bool silu = L.act != CBS_ACT_IDENTITY;
        auto kern = rk == 3 ? (silu ? stem_tc_rows_kernel<3, true> : stem_tc_rows_kernel<3, false>)
                            : (silu ? stem_tc_rows_kernel<1, true> : stem_tc_rows_kernel<1, false>);
        const cudaError_t e = set_max_dyn_smem(kern, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(kern, grid, kStemRowsThreads, (size_t)smem, s, tm, L, rg, status);
    }
    const int grid = std::min(g.n_tiles, L.grid);   // the plan's persistent CTAs
    const int n_mma = (L.Cout + 15) / 16 * 16;
    if (L.tf32)
        return L.out_nhwc ? launch_stem_tf32<true>(L, n_mma, g, grid, s, status)
                          : launch_stem_tf32<false>(L, n_mma, g, grid, s, status);
    const bool pairs = L.KS == 3 && L.stride == 2 && L.pad == 1 && (L.W & 1) == 0;
    if (L.out_nhwc)
        return pairs ? launch_stem_tc_as<true, true>(L, n_mma, g, grid, s, status)
                     : launch_stem_tc_as<true, false>(L, n_mma, g, grid, s, status);
    return pairs ? launch_stem_tc_as<false, true>(L, n_mma, g, grid, s, status)
                 : launch_stem_tc_as<false, false>(L, n_mma, g, grid, s, status);
}

}  // namespace

cudaError_t launch_stem(const StemLaunch &L, cudaStream_t s) {
    if (L.N == 0) return cudaSuccess;
    if (stem_uses_tensor_cores(L.tf32 ? 3 : L.kind, L.in_nhwc, L.c_pad, L.KS, L.Cout, (long long)L.N * L.OH * L.OW))
        return launch_stem_tc(L, s);
    switch (L.kind) {
        case 0: return launch_cout<0>(L, s);
        case 1: return launch_cout<1>(L, s);
        case 2: return launch_cout<2>(L, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace cbs
