// k_misc.cu -- setup and glue kernels: BN folding and weight packing, the
// chain-entry layout conversion, the upsample+concat neck glue, and the
// device status word that bounded waits report into.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "cbs_internal.cuh"
#include "tc_ptx.cuh"

namespace cbs {
namespace {

// ------------------------------------------------------------------ folding
// One CTA per output channel.  Float arithmetic is written with explicit
// round-to-nearest intrinsics so nothing is contracted into an FMA: the INT8
// codes, bias and scales must come out bit-identical to any other IEEE
// evaluation of the same steps.
//   s_c = gamma / sqrt(var + eps);   w' = w * s_c;   b' = beta - mean * s_c
// (with a conv bias cb:  b' = beta + (cb - mean) * s_c).
constexpr int kFoldThreads = 256;

__global__ void __launch_bounds__(kFoldThreads) fold_kernel(const FoldLaunch a) {
    const int co = blockIdx.x;
    const int KK = a.KS * a.KS;
    const int kin = a.C_in * KK;                 // OIHW row length
    const int kpad = KK * a.c_in_pad;            // packed row length (tap-major)
    const float s_c = __fdiv_rn(a.gamma[co], __fsqrt_rn(__fadd_rn(a.var[co], a.eps)));
    const float *wrow = a.w + (size_t)co * kin;

    float b_fold;
    if (a.conv_bias) {
        b_fold = __fadd_rn(a.beta[co], __fmul_rn(__fsub_rn(a.conv_bias[co], a.mean[co]), s_c));
    } else {
        b_fold = __fsub_rn(a.beta[co], __fmul_rn(a.mean[co], s_c));
    }

    if (a.variant == CBS_VARIANT_SIMT_FP32) {
        float *out = static_cast<float *>(a.w_packed);
        for (int k = threadIdx.x; k < kin; k += blockDim.x) {
            const int tap = k / a.C_in, ci = k - tap * a.C_in;
            out[(size_t)k * a.C_out + co] = __fmul_rn(wrow[ci * KK + tap], s_c);
        }
        if (threadIdx.x == 0) static_cast<float *>(a.bias)[co] = b_fold;
        return;
    }
    if (a.variant == CBS_VARIANT_TC_TF32X3) {
        // Head = w' with its low 13 mantissa bits cleared (a TF32 number) in
        // rows 0..C_out-1; tail = w' - head (exact) in rows C_out..2 C_out-1.
        float *out = static_cast<float *>(a.w_packed);
        for (int k = threadIdx.x; k < kpad; k += blockDim.x) {
            const int tap = k / a.c_in_pad, ci = k - tap * a.c_in_pad;
            const float v = ci < a.C_in ? __fmul_rn(wrow[ci * KK + tap], s_c) : 0.0f;
            const float head = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
            out[(size_t)co * kpad + k] = head;
            out[(size_t)(a.C_out + co) * kpad + k] = __fsub_rn(v, head);
        }
        if (threadIdx.x == 0) static_cast<float *>(a.bias)[co] = b_fold;
        return;
    }
    if (a.variant == CBS_VARIANT_TC_TF32 || a.variant == CBS_VARIANT_TC_BF16) {
        for (int k = threadIdx.x; k < kpad; k += blockDim.x) {
            const int tap = k / a.c_in_pad, ci = k - tap * a.c_in_pad;
            const float v = ci < a.C_in ? __fmul_rn(wrow[ci * KK + tap], s_c) : 0.0f;
            if (a.variant == CBS_VARIANT_TC_TF32)
                static_cast<float *>(a.w_packed)[(size_t)co * kpad + k] = v;
            else
                static_cast<__nv_bfloat16 *>(a.w_packed)[(size_t)co * kpad + k] = __float2bfloat16_rn(v);
        }
        if (threadIdx.x == 0) static_cast<float *>(a.bias)[co] = b_fold;
        return;
    }
    // INT8: per-channel symmetric scale s_w = max|w'| / 127.
    __shared__ float red[kFoldThreads / 32];
    float amax = 0.0f;
    for (int k = threadIdx.x; k < kin; k += blockDim.x)
        amax = fmaxf(amax, fabsf(__fmul_rn(wrow[k], s_c)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    float s_w = __fdiv_rn(amax, 127.0f);
    if (s_w == 0.0f) s_w = 1.0f;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.w_packed);
    for (int k = threadIdx.x; k < kpad; k += blockDim.x) {
        const int tap = k / a.c_in_pad, ci = k - tap * a.c_in_pad;
        float q = 0.0f;
        if (ci < a.C_in) {
            q = rintf(__fdiv_rn(__fmul_rn(wrow[ci * KK + tap], s_c), s_w));
            q = fminf(fmaxf(q, -127.0f), 127.0f);
        }
        out[(size_t)co * kpad + k] = __float2bfloat16_rn(q);  // exact: |q| <= 127
    }
    // Input zero point: the bias becomes bias_i32 - z_x * sum(q_w[c, :]),
    // in two's-complement int32 arithmetic (the kernels' sums are exact
    // modulo 2^32, so they are exact whenever the true accumulator fits).
    __shared__ unsigned int qsum_red[kFoldThreads / 32];
    unsigned int qsum = 0u;
    if (a.z_x != 0) {
        for (int k = threadIdx.x; k < kin; k += blockDim.x) {
            float q = rintf(__fdiv_rn(__fmul_rn(wrow[k], s_c), s_w));
            q = fminf(fmaxf(q, -127.0f), 127.0f);
            qsum += (unsigned int)(int)q;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qsum += __shfl_xor_sync(0xffffffffu, qsum, o);
        if ((threadIdx.x & 31) == 0) qsum_red[threadIdx.x >> 5] = qsum;
        __syncthreads();
        qsum = 0u;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) qsum += qsum_red[i];
    }
    if (threadIdx.x == 0) {
        const float mc = __fmul_rn(a.s_x, s_w);
        const float bq = rintf(__fdiv_rn(b_fold, mc));
        int32_t bi;
        if (bq >= 2147483648.0f) bi = INT32_MAX;
        else if (bq < -2147483648.0f) bi = INT32_MIN;
        else bi = (int32_t)bq;
        if (a.z_x != 0) bi = (int32_t)((unsigned int)bi - (unsigned int)a.z_x * qsum);
        static_cast<int32_t *>(a.bias)[co] = bi;
        a.m_c[co] = mc;
    }
}

// ------------------------------------------------------------ entry packing
// NCHW float -> NHWC (channels padded to c_pad with zeros) in float, bf16 or
// int8 (q = rne(clamp(x / s_x, -128, 127))).  32x32 (w, c) tiles through
// shared memory so both the read and the write are coalesced.
template <typename T>
__device__ __forceinline__ T convert_out(float v, float s_x, int zp);
template <>
__device__ __forceinline__ float convert_out<float>(float v, float, int) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 convert_out<__nv_bfloat16>(float v, float, int) {
    return __float2bfloat16_rn(v);
}
// q = clamp(rne(x / s_x) + zp, -128, 127); with zp = 0 the same as
// rne(clamp(x / s_x, -128, 127)) (integer bounds).
template <>
__device__ __forceinline__ int8_t convert_out<int8_t>(float v, float s_x, int zp) {
    float q = __fadd_rn(rintf(__fdiv_rn(v, s_x)), (float)zp);
    q = fminf(fmaxf(q, -128.0f), 127.0f);
    return (int8_t)q;
}
// Padding channels hold code 0 in every format.
template <typename T>
__device__ __forceinline__ T zero_code() { return convert_out<T>(0.0f, 1.0f, 0); }

template <typename T>
__global__ void pack_nhwc_kernel(const float *__restrict__ x, T *__restrict__ out, int C, int H,
                                 int W, int c_pad, float s_x, int zp) {
    __shared__ float tile[32][33];
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int w0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const int nh = blockIdx.z;  // n * H + h
    const int n = nh / H, h = nh - n * H;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, w = w0 + tx;
        float v = 0.0f;
        if (c < C && w < W) v = x[(((size_t)n * C + c) * H + h) * W + w];
        tile[i][tx] = v;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int w = w0 + i, c = c0 + tx;
        if (w < W && c < c_pad)
            out[(((size_t)n * H + h) * W + w) * c_pad + c] = c < C ? convert_out<T>(tile[tx][i], s_x, zp) : zero_code<T>();
    }
}

// Few channels (c_pad <= 8, e.g. a 3-channel frame padded to 4): one thread
// per pixel, each block a run of 128 pixels of a row, rows walked by a
// grid-stride loop.  Reads are coalesced per channel plane; a pixel's 4
// channels leave as one vector store.
template <typename T>
__device__ __forceinline__ void store4(T *dst, const T (&v)[8]);
template <>
__device__ __forceinline__ void store4<float>(float *dst, const float (&v)[8]) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, const __nv_bfloat16 (&v)[8]) {
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(v[0]) | ((uint32_t)__bfloat16_as_ushort(v[1]) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(v[2]) | ((uint32_t)__bfloat16_as_ushort(v[3]) << 16);
    *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
}
template <>
__device__ __forceinline__ void store4<int8_t>(int8_t *dst, const int8_t (&v)[8]) {
    *reinterpret_cast<uint32_t *>(dst) = (uint32_t)(uint8_t)v[0] | ((uint32_t)(uint8_t)v[1] << 8) |
                                         ((uint32_t)(uint8_t)v[2] << 16) | ((uint32_t)(uint8_t)v[3] << 24);
}

constexpr int kPackSmallThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kPackSmallThreads) pack_nhwc_small_kernel(const float *__restrict__ x,
                                                                            T *__restrict__ out, int C, int H, int W,
                                                                            int rows, int c_pad, float s_x, int zp) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int w = blockIdx.x * kPackSmallThreads + threadIdx.x;
    if (w >= W) return;
    const size_t hw = (size_t)H * W;
    for (int row = blockIdx.y; row < rows; row += gridDim.y) {   // row = n * H + h
        const int n = row / H, h = row - n * H;
        const float *src = x + (size_t)n * C * hw + (size_t)h * W + w;
        T v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = c < C ? convert_out<T>(__ldg(src + c * hw), s_x, zp) : zero_code<T>();
        T *dst = out + ((size_t)row * W + w) * c_pad;
        if (c_pad == 4) {
            store4<T>(dst, v);
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                if (c < c_pad) dst[c] = v[c];
        }
    }
}

// Four consecutive pixels of 4 padded channels, packed into 16, 32 or 64
// contiguous output bytes.
template <typename T>
__device__ __forceinline__ void store16(T *dst, const T (&v)[16]);
template <>
__device__ __forceinline__ void store16<float>(float *dst, const float (&v)[16]) {
#pragma unroll
    for (int p = 0; p < 4; ++p)
        reinterpret_cast<float4 *>(dst)[p] = make_float4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
}
template <>
__device__ __forceinline__ void store16<__nv_bfloat16>(__nv_bfloat16 *dst, const __nv_bfloat16 (&v)[16]) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        w[k] = (uint32_t)__bfloat16_as_ushort(v[2 * k]) | ((uint32_t)__bfloat16_as_ushort(v[2 * k + 1]) << 16);
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}
template <>
__device__ __forceinline__ void store16<int8_t>(int8_t *dst, const int8_t (&v)[16]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = (uint32_t)(uint8_t)v[4 * k] | ((uint32_t)(uint8_t)v[4 * k + 1] << 8) |
               ((uint32_t)(uint8_t)v[4 * k + 2] << 16) | ((uint32_t)(uint8_t)v[4 * k + 3] << 24);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float lane_of(const float4 &v, int p) {
    return p == 0 ? v.x : (p == 1 ? v.y : (p == 2 ? v.z : v.w));
}

// pack_nhwc_small_kernel for 4 padded channels and W a multiple of 4: four
// pixels per thread, one 16-byte load per input plane and 16-64 contiguous
// output bytes, so each thread keeps several wide loads in flight.
template <typename T>
__global__ void __launch_bounds__(kPackSmallThreads) pack_nhwc_quad_kernel(const float *__restrict__ x,
                                                                           T *__restrict__ out, int C, int H, int W,
                                                                           int rows, float s_x, int zp) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int w4 = blockIdx.x * kPackSmallThreads + threadIdx.x;   // quad of pixels 4 w4 .. 4 w4 + 3
    if (w4 >= (W >> 2)) return;
    const size_t hw = (size_t)H * W;   // a multiple of 4
    for (int row = blockIdx.y; row < rows; row += gridDim.y) {   // row = n * H + h
        const int n = row / H, h = row - n * H;
        const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)n * C * hw + (size_t)h * W) + w4;
        float4 pl[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) pl[c] = c < C ? __ldg(src + c * (hw >> 2)) : make_float4(0.f, 0.f, 0.f, 0.f);
        T v[16];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int c = 0; c < 4; ++c) v[4 * p + c] = c < C ? convert_out<T>(lane_of(pl[c], p), s_x, zp) : zero_code<T>();
        store16<T>(out + ((size_t)row * W + 4 * (size_t)w4) * 4, v);
    }
}

template <typename T>
__global__ void pack_nchw_kernel(const float *__restrict__ x, T *__restrict__ out, size_t count,
                                 float s_x, int zp) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count;
         i += (size_t)gridDim.x * blockDim.x)
        out[i] = convert_out<T>(x[i], s_x, zp);
}

// ------------------------------------------------------------------- glue
// NHWC, 16-byte vectors: out[n,h,w,:] = [a[n,h/2,w/2,:], b[n,h,w,:]].
__global__ void upcat_nhwc_vec_kernel(const uint4 *__restrict__ a, int va, const uint4 *__restrict__ b,
                                      int vb, uint4 *__restrict__ out, int n, int h, int w) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int vt = va + vb;
    const size_t total = (size_t)n * h * w * vt;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int v = (int)(i % vt);
        const size_t pix = i / vt;
        const int x = (int)(pix % w);
        const size_t nhh = pix / w;
        const int y = (int)(nhh % h);
        const int img = (int)(nhh / h);
        uint4 val;
        if (v < va)
            val = a[(((size_t)img * (h / 2) + y / 2) * (w / 2) + x / 2) * va + v];
        else
            val = b[pix * vb + (v - va)];
        out[i] = val;
    }
}

template <typename T>
__global__ void upcat_elem_kernel(const T *__restrict__ a, int ca, const T *__restrict__ b, int cb,
                                  T *__restrict__ out, int n, int h, int w, int nhwc) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int ct = ca + cb;
    const size_t total = (size_t)n * h * w * ct;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        int c, x, y, img;
        if (nhwc) {
            c = (int)(i % ct);
            size_t r = i / ct;
            x = (int)(r % w); r /= w;
            y = (int)(r % h); img = (int)(r / h);
        } else {
            x = (int)(i % w);
            size_t r = i / w;
            y = (int)(r % h); r /= h;
            c = (int)(r % ct); img = (int)(r / ct);
        }
        T val;
        if (c < ca) {
            const int ys = y / 2, xs = x / 2;
            val = nhwc ? a[(((size_t)img * (h / 2) + ys) * (w / 2) + xs) * ca + c]
                       : a[(((size_t)img * ca + c) * (h / 2) + ys) * (w / 2) + xs];
        } else {
            const int cc = c - ca;
            val = nhwc ? b[(((size_t)img * h + y) * w + x) * cb + cc]
                       : b[(((size_t)img * cb + cc) * h + y) * w + x];
        }
        out[i] = val;
    }
}

// 2-D max pooling ("YOLO26N Inference Optimisation": maxpool2d, three per
// frame in SPPF): the window's positions inside the image only, floor output
// size, a NaN in the window gives NaN.  One thread per output element in the
// tensor's own order, so NHWC reads of a window position are coalesced over
// channels.  int8 codes compare like their values (the scale is positive).
template <typename T>
__device__ __forceinline__ bool pool_is_nan(T v) { return false; }
template <>
__device__ __forceinline__ bool pool_is_nan<float>(float v) { return v != v; }
template <>
__device__ __forceinline__ bool pool_is_nan<__nv_bfloat16>(__nv_bfloat16 v) {
    return (__bfloat16_as_ushort(v) & 0x7fffu) > 0x7f80u;
}
template <typename T>
__device__ __forceinline__ bool pool_greater(T a, T b) { return a > b; }
template <>
__device__ __forceinline__ bool pool_greater<__nv_bfloat16>(__nv_bfloat16 a, __nv_bfloat16 b) {
    return __bfloat162float(a) > __bfloat162float(b);
}

template <typename T>
__global__ void maxpool_kernel(const T *__restrict__ x, T *__restrict__ y, int N, int C, int H, int W, int OH,
                               int OW, int k, int stride, int pad, int nhwc) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const size_t total = (size_t)N * C * OH * OW;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        int n, c, oh, ow;
        if (nhwc) {
            c = (int)(i % C);
            size_t r = i / C;
            ow = (int)(r % OW);
            r /= OW;
            oh = (int)(r % OH);
            n = (int)(r / OH);
        } else {
            ow = (int)(i % OW);
            size_t r = i / OW;
            oh = (int)(r % OH);
            r /= OH;
            c = (int)(r % C);
            n = (int)(r / C);
        }
        T m = T(0), nanv = T(0);
        bool any = false, nan = false;
        for (int r = 0; r < k; ++r) {
            const int ih = oh * stride - pad + r;
            if (ih < 0 || ih >= H) continue;
            for (int s = 0; s < k; ++s) {
                const int iw = ow * stride - pad + s;
                if (iw < 0 || iw >= W) continue;
                const T v = nhwc ? x[(((size_t)n * H + ih) * W + iw) * C + c] : x[(((size_t)n * C + c) * H + ih) * W + iw];
                if (pool_is_nan<T>(v)) {
                    nan = true;
                    nanv = v;
                } else if (!any || pool_greater<T>(v, m)) {
                    m = v;
                    any = true;
                }
            }
        }
        y[i] = nan ? nanv : m;
    }
}

// ---------------------------------------------------------------- SPPF pools
// y = concat(p(x), p(p(x)), p(p(p(x)))) along channels, p = the k x k max
// pool with stride 1 and padding k/2 whose padded positions take no part (the
// SPPF block's three chained pools; "YOLO26N Inference Optimisation", kernel
// profile: maxpool2d, three per frame).  One CTA per (16x16 output tile,
// image, group of kSppfCg channels) keeps the tile with a halo of 3 (k/2) in
// shared memory.  Positions outside the image hold the type's lowest value:
// every window holds its own in-image centre, so the lowest value never wins
// over a real one and the max equals the max over the in-image positions.
// Each pool is a horizontal, then a vertical running max in shared memory;
// the region it covers shrinks by k/2 per pool, and after each pool the
// tile's interior goes to its channel slice of y.  A NaN in a window gives NaN.
constexpr int kSppfTile = 16;

template <typename T>
struct PoolOps;
template <>
struct PoolOps<float> {
    static __device__ __forceinline__ float lowest() { return __int_as_float(0xff800000); }   // -inf
    static __device__ __forceinline__ float mx(float a, float b) {
        return a != a ? a : (b != b ? b : (a > b ? a : b));
    }
};
template <>
struct PoolOps<__nv_bfloat16> {
    static __device__ __forceinline__ __nv_bfloat16 lowest() { return __ushort_as_bfloat16(0xff80); }   // -inf
    static __device__ __forceinline__ bool nan(__nv_bfloat16 v) { return (__bfloat16_as_ushort(v) & 0x7fffu) > 0x7f80u; }
    static __device__ __forceinline__ __nv_bfloat16 mx(__nv_bfloat16 a, __nv_bfloat16 b) {
        return nan(a) ? a : (nan(b) ? b : (__bfloat162float(a) > __bfloat162float(b) ? a : b));
    }
};
template <>
struct PoolOps<int8_t> {
    static __device__ __forceinline__ int8_t lowest() { return (int8_t)-128; }
    static __device__ __forceinline__ int8_t mx(int8_t a, int8_t b) { return a > b ? a : b; }
};

template <typename T>
__global__ void __launch_bounds__(256) sppf_pool_kernel(const T *__restrict__ x, T *__restrict__ y, int N, int C,
                                                        int H, int W, int hk, int cg, int tiles_w, int nhwc) {
    extern __shared__ __align__(16) uint8_t sppf_smem[];
    using O = PoolOps<T>;
    const int R = 3 * hk, S = kSppfTile + 2 * R;
    T *buf = reinterpret_cast<T *>(sppf_smem);
    T *tmp = buf + (size_t)S * S * cg;
    const int n = blockIdx.y;
    const int c0 = blockIdx.z * cg;
    const int oh0 = (blockIdx.x / tiles_w) * kSppfTile, ow0 = (blockIdx.x % tiles_w) * kSppfTile;
    const int C3 = 3 * C;
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    // The tile and its halo; the lowest value outside the image and past C.
    for (int e = threadIdx.x; e < S * S * cg; e += blockDim.x) {
        const int c = e % cg, pos = e / cg;
        const int ih = oh0 - R + pos / S, iw = ow0 - R + pos % S;
        T v = O::lowest();
        if (ih >= 0 && ih < H && iw >= 0 && iw < W && c0 + c < C)
            v = nhwc ? x[(((size_t)n * H + ih) * W + iw) * C + c0 + c] : x[(((size_t)n * C + c0 + c) * H + ih) * W + iw];
        buf[e] = v;
    }
    __syncthreads();
    for (int r = 1; r <= 3; ++r) {
        const int ext = (3 - r) * hk;
        // Horizontal max over rows [R-ext-hk, R+T+ext+hk) and columns [R-ext, R+T+ext).
        {
            const int y0 = R - ext - hk, ny = kSppfTile + 2 * (ext + hk);
            const int x0 = R - ext, nx = kSppfTile + 2 * ext;
            for (int e = threadIdx.x; e < ny * nx * cg; e += blockDim.x) {
                const int c = e % cg, pos = e / cg;
                const int yy = y0 + pos / nx, xx = x0 + pos % nx;
                const T *row = buf + ((size_t)yy * S) * cg + c;
                T v = row[(size_t)(xx - hk) * cg];
                for (int dx = -hk + 1; dx <= hk; ++dx) v = O::mx(v, row[(size_t)(xx + dx) * cg]);
                tmp[((size_t)yy * S + xx) * cg + c] = v;
            }
        }
        __syncthreads();
        // Vertical max into buf over rows and columns [R-ext, R+T+ext).
        {
            const int y0 = R - ext, nyx = kSppfTile + 2 * ext;
            for (int e = threadIdx.x; e < nyx * nyx * cg; e += blockDim.x) {
                const int c = e % cg, pos = e / cg;
                const int yy = y0 + pos / nyx, xx = y0 + pos % nyx;
                const int ih = oh0 - R + yy, iw = ow0 - R + xx;
                T v = O::lowest();
                if (ih >= 0 && ih < H && iw >= 0 && iw < W) {
                    const T *col = tmp + (size_t)xx * cg + c;
                    v = col[(size_t)(yy - hk) * S * cg];
                    for (int dy = -hk + 1; dy <= hk; ++dy) v = O::mx(v, col[(size_t)(yy + dy) * S * cg]);
                }
                buf[((size_t)yy * S + xx) * cg + c] = v;
            }
        }
        __syncthreads();
        // Pool r over the tile's interior to channel slice r - 1 of y.
        for (int e = threadIdx.x; e < kSppfTile * kSppfTile * cg; e += blockDim.x) {
            const int c = e % cg, pos = e / cg;
            const int oh = oh0 + pos / kSppfTile, ow = ow0 + pos % kSppfTile;
            if (oh >= H || ow >= W || c0 + c >= C) continue;
            const T v = buf[((size_t)(R + pos / kSppfTile) * S + R + pos % kSppfTile) * cg + c];
            const int ch = (r - 1) * C + c0 + c;
            if (nhwc) y[(((size_t)n * H + oh) * W + ow) * C3 + ch] = v;
            else y[(((size_t)n * C3 + ch) * H + oh) * W + ow] = v;
        }
        // The next pool's horizontal pass reads buf, which these writes only read.
    }
}

__device__ unsigned int g_cbs_status_word;

// Diagnostic for the timeout path: thread 0 waits, through the same bounded
// mbarrier wait the tensor-core kernels use, on a barrier that nothing
// arrives at.  After limit_ns the wait gives up and the kernel records a
// timeout in the status word, as a kernel does when one of its waits runs out.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, unsigned int *status) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait_bounded(b, 0, limit_ns)) atomicOr(status, 1u);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
    unsigned int *status = device_status_word();
    if (!status) return cudaErrorInvalidValue;
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
    return cudaGetLastError();
}

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

cbs_status current_context_id(unsigned long long *id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        void *p1 = nullptr, *p2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 12000, cudaEnableDefault, &q1) ==
                cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(p1);
            get_id = reinterpret_cast<CtxGetIdFn>(p2);
        }
    });
    if (!get_current || !get_id) return fail(CBS_ERR_CUDA, "driver entry points cuCtxGetCurrent/cuCtxGetId unavailable");
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuCtxGetCurrent failed");
    *id = 0;
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuCtxGetId failed");
    return CBS_OK;
}

int current_device_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kDefaultNumSMs;
    if (cached[dev] <= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return kDefaultNumSMs;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

int grid_for(size_t count, int threads) {
    size_t blocks = (count + threads - 1) / threads;
    const size_t cap = (size_t)current_device_sms() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

}  // namespace

cudaError_t launch_fold(const FoldLaunch &L, cudaStream_t s) {
    fold_kernel<<<L.C_out, kFoldThreads, 0, s>>>(L);   // set-up: a plain launch, fully ordered
    return cudaGetLastError();
}

cudaError_t launch_pack_input(const float *x, void *out, int N, int C, int H, int W, int c_pad,
                              int to_nhwc, int dtype, float s_x, int zp, cudaStream_t s) {
    if (to_nhwc && c_pad == 4 && W % 4 == 0) {   // x and out are 16-byte aligned (checked by the caller)
        const int gx = (W / 4 + kPackSmallThreads - 1) / kPackSmallThreads;
        const int rows = N * H;
        int gy = current_device_sms() * 32 / gx;
        gy = gy < 1 ? 1 : (gy > rows ? rows : (gy > 65535 ? 65535 : gy));
        const dim3 grid(gx, gy);
        if (dtype == 0) launch_kernel(pack_nhwc_quad_kernel<float>, grid, kPackSmallThreads, 0, s, x, (float *)out, C, H, W, rows, s_x, zp);
        else if (dtype == 1) launch_kernel(pack_nhwc_quad_kernel<__nv_bfloat16>, grid, kPackSmallThreads, 0, s, x, (__nv_bfloat16 *)out, C, H, W, rows, s_x, zp);
        else launch_kernel(pack_nhwc_quad_kernel<int8_t>, grid, kPackSmallThreads, 0, s, x, (int8_t *)out, C, H, W, rows, s_x, zp);
    } else if (to_nhwc && c_pad <= 8) {
        const int gx = (W + kPackSmallThreads - 1) / kPackSmallThreads;
        const int rows = N * H;
        int gy = current_device_sms() * 32 / gx;
        gy = gy < 1 ? 1 : (gy > rows ? rows : (gy > 65535 ? 65535 : gy));
        const dim3 grid(gx, gy);
        if (dtype == 0) launch_kernel(pack_nhwc_small_kernel<float>, grid, kPackSmallThreads, 0, s, x, (float *)out, C, H, W, rows, c_pad, s_x, zp);
        else if (dtype == 1) launch_kernel(pack_nhwc_small_kernel<__nv_bfloat16>, grid, kPackSmallThreads, 0, s, x, (__nv_bfloat16 *)out, C, H, W, rows, c_pad, s_x, zp);
        else launch_kernel(pack_nhwc_small_kernel<int8_t>, grid, kPackSmallThreads, 0, s, x, (int8_t *)out, C, H, W, rows, c_pad, s_x, zp);
    } else if (to_nhwc) {
        dim3 grid((W + 31) / 32, (c_pad + 31) / 32, N * H), block(32, 8);
        if (dtype == 0) launch_kernel(pack_nhwc_kernel<float>, grid, block, 0, s, x, (float *)out, C, H, W, c_pad, s_x, zp);
        else if (dtype == 1) launch_kernel(pack_nhwc_kernel<__nv_bfloat16>, grid, block, 0, s, x, (__nv_bfloat16 *)out, C, H, W, c_pad, s_x, zp);
        else launch_kernel(pack_nhwc_kernel<int8_t>, grid, block, 0, s, x, (int8_t *)out, C, H, W, c_pad, s_x, zp);
    } else {
        const size_t count = (size_t)N * C * H * W;
        const int g = grid_for(count, 256);
        if (dtype == 0) launch_kernel(pack_nchw_kernel<float>, g, 256, 0, s, x, (float *)out, count, s_x, zp);
        else if (dtype == 1) launch_kernel(pack_nchw_kernel<__nv_bfloat16>, g, 256, 0, s, x, (__nv_bfloat16 *)out, count, s_x, zp);
        else launch_kernel(pack_nchw_kernel<int8_t>, g, 256, 0, s, x, (int8_t *)out, count, s_x, zp);
    }
    return cudaGetLastError();
}

cudaError_t launch_upsample_concat(const void *a, int ca, const void *b, int cb, void *out, int n,
                                   int h, int w, int nhwc, int eb, cudaStream_t s) {
    const bool vec = nhwc && (ca * eb) % 16 == 0 && (cb * eb) % 16 == 0 &&
                     aligned16(a) && aligned16(b) && aligned16(out);
    if (vec) {
        const int va = ca * eb / 16, vb = cb * eb / 16;
        const size_t total = (size_t)n * h * w * (va + vb);
        launch_kernel(upcat_nhwc_vec_kernel, grid_for(total, 256), 256, 0, s, 
            (const uint4 *)a, va, (const uint4 *)b, vb, (uint4 *)out, n, h, w);
    } else {
        const size_t total = (size_t)n * h * w * (ca + cb);
        const int g = grid_for(total, 256);
        if (eb == 4) launch_kernel(upcat_elem_kernel<uint32_t>, g, 256, 0, s, (const uint32_t *)a, ca, (const uint32_t *)b, cb, (uint32_t *)out, n, h, w, nhwc);
        else if (eb == 2) launch_kernel(upcat_elem_kernel<uint16_t>, g, 256, 0, s, (const uint16_t *)a, ca, (const uint16_t *)b, cb, (uint16_t *)out, n, h, w, nhwc);
        else launch_kernel(upcat_elem_kernel<uint8_t>, g, 256, 0, s, (const uint8_t *)a, ca, (const uint8_t *)b, cb, (uint8_t *)out, n, h, w, nhwc);
    }
    return cudaGetLastError();
}

cudaError_t launch_maxpool(const void *x, void *y, int n, int c, int h, int w, int k, int stride, int pad, int nhwc,
                           int eb, cudaStream_t s) {
    const int oh = (h + 2 * pad - k) / stride + 1, ow = (w + 2 * pad - k) / stride + 1;
    const int g = grid_for((size_t)n * c * oh * ow, 256);
    if (eb == 4)
        return launch_kernel(maxpool_kernel<float>, g, 256, 0, s, (const float *)x, (float *)y, n, c, h, w, oh, ow, k,
                             stride, pad, nhwc);
    if (eb == 2)
        return launch_kernel(maxpool_kernel<__nv_bfloat16>, g, 256, 0, s, (const __nv_bfloat16 *)x, (__nv_bfloat16 *)y,
                             n, c, h, w, oh, ow, k, stride, pad, nhwc);
    return launch_kernel(maxpool_kernel<int8_t>, g, 256, 0, s, (const int8_t *)x, (int8_t *)y, n, c, h, w, oh, ow, k,
                         stride, pad, nhwc);
}

cudaError_t launch_sppf_pool(const void *x, void *y, int n, int c, int h, int w, int k, int nhwc, int eb,
                             cudaStream_t s) {
    const int hk = k / 2, S = kSppfTile + 6 * hk;
    // Channels per CTA: 32 bytes of each pixel; two S x S buffers in shared memory.
    const int cg = 32 / eb;
    const int smem = 2 * S * S * cg * eb;
    const int tiles_w = (w + kSppfTile - 1) / kSppfTile, tiles_h = (h + kSppfTile - 1) / kSppfTile;
    const dim3 grid(tiles_w * tiles_h, n, (c + cg - 1) / cg);
    if (grid.z > 65535 || n > 65535) return cudaErrorInvalidValue;
    cudaError_t e;
    if (eb == 4) {
        if ((e = set_max_dyn_smem(sppf_pool_kernel<float>, smem)) != cudaSuccess) return e;
        return launch_kernel(sppf_pool_kernel<float>, grid, 256, smem, s, (const float *)x, (float *)y, n, c, h, w,
                             hk, cg, tiles_w, nhwc);
    }
    if (eb == 2) {
        if ((e = set_max_dyn_smem(sppf_pool_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        return launch_kernel(sppf_pool_kernel<__nv_bfloat16>, grid, 256, smem, s, (const __nv_bfloat16 *)x,
                             (__nv_bfloat16 *)y, n, c, h, w, hk, cg, tiles_w, nhwc);
    }
    if ((e = set_max_dyn_smem(sppf_pool_kernel<int8_t>, smem)) != cudaSuccess) return e;
    return launch_kernel(sppf_pool_kernel<int8_t>, grid, 256, smem, s, (const int8_t *)x, (int8_t *)y, n, c, h, w, hk,
                         cg, tiles_w, nhwc);
}

unsigned int *device_status_word() {
    // One address per device and context: looked up again after a device
    // reset (the module, and the word with it, is then loaded afresh).
    static unsigned int *cache[64] = {nullptr};
    static unsigned long long cache_ctx[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != CBS_OK) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev] || ctx == 0 || cache_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_cbs_status_word) != cudaSuccess) return nullptr;
        if (current_context_id(&ctx) != CBS_OK) return nullptr;
        cache[dev] = static_cast<unsigned int *>(p);
        cache_ctx[dev] = ctx;
    }
    return cache[dev];
}

cbs_status read_and_reset_status(int *status_out, int reset, cudaStream_t s) {
    unsigned int v = 0;
    cbs_status st = cuda_check(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (st != CBS_OK) return st;
    st = cuda_check(cudaMemcpyFromSymbol(&v, g_cbs_status_word, sizeof(v)), "read status word");
    if (st != CBS_OK) return st;
    if (reset) {
        const unsigned int zero = 0;
        st = cuda_check(cudaMemcpyToSymbol(g_cbs_status_word, &zero, sizeof(zero)), "reset status word");
        if (st != CBS_OK) return st;
    }
    *status_out = v ? (int)CBS_ERR_TIMEOUT : (int)CBS_OK;
    return CBS_OK;
}

}  // namespace cbs
