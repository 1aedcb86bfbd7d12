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
// profile: maxpool2d, three per frame).  One CTA per (output tile of up to
// 32 x 32, image, group of 32 bytes of channels) keeps the tile with a halo of
// 3 (k/2) in shared memory.  Positions outside the image hold the type's
// lowest value: every window holds its own in-image centre, so the lowest
// value never wins over a real one and the max equals the max over the
// in-image positions.  Each pool is a horizontal, then a vertical running
// max in shared memory over a region that shrinks by k/2 per pool; after
// each pool the tile's interior goes to its channel slice of y.  A NaN in a
// window gives NaN.  Rows are spread over the warps and (column, channel)
// pairs over the lanes, so no index needs a division by a runtime value.
constexpr int kSppfMaxTile = 32;

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

// Max of two 16-byte vectors of T, element by element (NaN-propagating for
// the float types); the vector of lowest values.
template <typename T>
struct VecPool;
template <>
struct VecPool<float> {
    static __device__ __forceinline__ uint4 lowest() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
    static __device__ __forceinline__ uint32_t m1(uint32_t a, uint32_t b) {
        return __float_as_uint(PoolOps<float>::mx(__uint_as_float(a), __uint_as_float(b)));
    }
    static __device__ __forceinline__ uint4 mx(uint4 a, uint4 b) {
        return make_uint4(m1(a.x, b.x), m1(a.y, b.y), m1(a.z, b.z), m1(a.w, b.w));
    }
};
template <>
struct VecPool<__nv_bfloat16> {
    static __device__ __forceinline__ uint4 lowest() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
    static __device__ __forceinline__ uint32_t m1(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    static __device__ __forceinline__ uint4 mx(uint4 a, uint4 b) {
        return make_uint4(m1(a.x, b.x), m1(a.y, b.y), m1(a.z, b.z), m1(a.w, b.w));
    }
};
template <>
struct VecPool<int8_t> {
    static __device__ __forceinline__ uint4 lowest() { return make_uint4(0x80808080u, 0x80808080u, 0x80808080u, 0x80808080u); }
    static __device__ __forceinline__ uint4 mx(uint4 a, uint4 b) {
        return make_uint4(__vmaxs4(a.x, b.x), __vmaxs4(a.y, b.y), __vmaxs4(a.z, b.z), __vmaxs4(a.w, b.w));
    }
};

// Shared memory holds, per position of the tile and its halo, the CTA's 32
// bytes of channels as two 16-byte vectors.  Global memory is read and
// written in 16-byte vectors where a pixel's channels are 16-byte multiples
// (NHWC with C * sizeof(T) a multiple of 16), element by element otherwise.
template <typename T, int HK>
__global__ void __launch_bounds__(256) sppf_pool_kernel(const T *__restrict__ x, T *__restrict__ y, int N, int C,
                                                        int H, int W, int TH, int TW, int tiles_w, int nhwc) {
    extern __shared__ __align__(16) uint8_t sppf_smem[];
    using V = VecPool<T>;
    constexpr int VE = 16 / (int)sizeof(T);   // elements per 16-byte vector
    constexpr int CG = 2 * VE;                // channels per CTA
    constexpr int R = 3 * HK;
    const int SH = TH + 2 * R, SW = TW + 2 * R;
    uint4 *buf = reinterpret_cast<uint4 *>(sppf_smem);
    uint4 *tmp = buf + (size_t)SH * SW * 2;
    const int n = blockIdx.y;
    const int c0 = blockIdx.z * CG;
    const int oh0 = (blockIdx.x / tiles_w) * TH, ow0 = (blockIdx.x % tiles_w) * TW;
    const int C3 = 3 * C;
    const bool vec = nhwc && (C * (int)sizeof(T)) % 16 == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    // The tile and its halo; the lowest value outside the image and past C.
    for (int yy = warp; yy < SH; yy += nwarps) {
        const int ih = oh0 - R + yy;
        for (int i = lane; i < SW * 2; i += 32) {
            const int xx = i >> 1, v = i & 1;
            const int iw = ow0 - R + xx;
            const int cv = c0 + v * VE;
            uint4 val = V::lowest();
            if (ih >= 0 && ih < H && iw >= 0 && iw < W && cv < C) {
                if (vec) {
                    val = __ldg(reinterpret_cast<const uint4 *>(x + (((size_t)n * H + ih) * W + iw) * C + cv));
                } else {
                    T e[VE];
                    const T *lw = reinterpret_cast<const T *>(&val);
#pragma unroll
                    for (int j = 0; j < VE; ++j)
                        e[j] = cv + j < C ? (nhwc ? x[(((size_t)n * H + ih) * W + iw) * C + cv + j]
                                                  : x[(((size_t)n * C + cv + j) * H + ih) * W + iw])
                                          : lw[j];
                    val = *reinterpret_cast<const uint4 *>(e);
                }
            }
            buf[(size_t)yy * SW * 2 + i] = val;
        }
    }
    __syncthreads();
#pragma unroll 1
    for (int r = 1; r <= 3; ++r) {
        const int ext = (3 - r) * HK;
        // Horizontal max over rows [R-ext-HK, R+TH+ext+HK) and columns [R-ext, R+TW+ext).
        const int hx0 = R - ext, hnx = TW + 2 * ext;
        for (int yy = R - ext - HK + warp; yy < R + TH + ext + HK; yy += nwarps) {
            const uint4 *row = buf + (size_t)yy * SW * 2;
            uint4 *trow = tmp + (size_t)yy * SW * 2;
            for (int i = lane; i < hnx * 2; i += 32) {
                const int j = hx0 * 2 + i;   // (column, vector) index within the row
                uint4 m = row[j - 2 * HK];
#pragma unroll
                for (int dx = -HK + 1; dx <= HK; ++dx) m = V::mx(m, row[j + 2 * dx]);
                trow[j] = m;
            }
        }
        __syncthreads();
        // Vertical max into buf over rows and columns [R-ext, R+T+ext); the lowest
        // value outside the image.
        for (int yy = R - ext + warp; yy < R + TH + ext; yy += nwarps) {
            const int ih = oh0 - R + yy;
            uint4 *brow = buf + (size_t)yy * SW * 2;
            for (int i = lane; i < hnx * 2; i += 32) {
                const int j = hx0 * 2 + i;
                const int iw = ow0 - R + (j >> 1);
                uint4 m = V::lowest();
                if (ih >= 0 && ih < H && iw >= 0 && iw < W) {
                    const uint4 *col = tmp + j;
                    m = col[(size_t)(yy - HK) * SW * 2];
#pragma unroll
                    for (int dy = -HK + 1; dy <= HK; ++dy) m = V::mx(m, col[(size_t)(yy + dy) * SW * 2]);
                }
                brow[j] = m;
            }
        }
        __syncthreads();
        // Pool r over the tile's interior to channel slice r - 1 of y (the next
        // pool's horizontal pass only reads buf as well).
        for (int ty = warp; ty < TH; ty += nwarps) {
            const int oh = oh0 + ty;
            if (oh >= H) break;
            const uint4 *brow = buf + (size_t)(R + ty) * SW * 2;
            for (int i = lane; i < TW * 2; i += 32) {
                const int tx = i >> 1, v = i & 1;
                const int ow = ow0 + tx;
                const int cv = c0 + v * VE;
                if (ow >= W || cv >= C) continue;
                const uint4 val = brow[(R + tx) * 2 + v];
                const int ch = (r - 1) * C + cv;
                if (vec) {
                    *reinterpret_cast<uint4 *>(y + (((size_t)n * H + oh) * W + ow) * C3 + ch) = val;
                } else {
                    const T *e = reinterpret_cast<const T *>(&val);
#pragma unroll
                    for (int j = 0; j < VE; ++j) {
                        if (cv + j >= C) break;
                        if (nhwc) y[(((size_t)n * H + oh) * W + ow) * C3 + ch + j] = e[j];
                        else y[(((size_t)n * C3 + ch + j) * H + oh) * W + ow] = e[j];
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------ INT8 seams
// Between an INT8 layer and a layer kept in float ("Edge optimisation of
// YOLO26", Highlights: sensitive layers stay in float), in the affine scheme
// r = s (q - z):
//   dequantise: r = (float)(q - z) * s, one IEEE multiply, then (BF16) the
//               round-to-nearest-even conversion;
//   quantise:   q = clamp(rne(x / s) + z, -128, 127), IEEE division (the
//               quantiser of the chain's entry packing).
// Elementwise over count values; 16 codes per thread (16-byte code vectors),
// the last ragged group element by element.
template <typename TO>
__device__ __forceinline__ void store_deq(TO *out, size_t i, float v);
template <>
__device__ __forceinline__ void store_deq<float>(float *out, size_t i, float v) { out[i] = v; }
template <>
__device__ __forceinline__ void store_deq<__nv_bfloat16>(__nv_bfloat16 *out, size_t i, float v) {
    out[i] = __float2bfloat16_rn(v);
}

template <typename TO>
__global__ void dequantize_i8_kernel(const int8_t *__restrict__ q, TO *__restrict__ out, size_t count, float s, int z) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const size_t groups = (count + 15) / 16;
    for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < groups; g += (size_t)gridDim.x * blockDim.x) {
        const size_t i0 = g * 16;
        if (i0 + 16 <= count) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(q + i0));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int code = (int)(int8_t)(ws[j >> 2] >> (8 * (j & 3)));
                store_deq<TO>(out, i0 + j, __fmul_rn((float)(code - z), s));
            }
        } else {
            for (size_t i = i0; i < count; ++i) store_deq<TO>(out, i, __fmul_rn((float)((int)q[i] - z), s));
        }
    }
}

template <typename TI>
__device__ __forceinline__ float load_val(const TI *x, size_t i);
template <>
__device__ __forceinline__ float load_val<float>(const float *x, size_t i) { return x[i]; }
template <>
__device__ __forceinline__ float load_val<__nv_bfloat16>(const __nv_bfloat16 *x, size_t i) {
    return __bfloat162float(x[i]);
}

template <typename TI>
__global__ void quantize_i8_kernel(const TI *__restrict__ x, int8_t *__restrict__ q, size_t count, float s, int z) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const size_t groups = (count + 15) / 16;
    for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < groups; g += (size_t)gridDim.x * blockDim.x) {
        const size_t i0 = g * 16;
        const int n = i0 + 16 <= count ? 16 : (int)(count - i0);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        for (int j = 0; j < n; ++j) {
            float v = __fadd_rn(rintf(__fdiv_rn(load_val<TI>(x, i0 + j), s)), (float)z);
            v = fminf(fmaxf(v, -128.0f), 127.0f);
            w[j >> 2] |= (uint32_t)(uint8_t)(int8_t)v << (8 * (j & 3));
        }
        if (n == 16) {
            *reinterpret_cast<uint4 *>(q + i0) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            for (int j = 0; j < n; ++j) q[i0 + j] = (int8_t)(w[j >> 2] >> (8 * (j & 3)));
        }
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

template <typename T>
cudaError_t launch_sppf_typed(const void *x, void *y, int n, int c, int h, int w, int hk, int nhwc, cudaStream_t s) {
    // Output tile: the whole image up to 32 x 32 (a 20x20 map is one tile).
    const int th = h < kSppfMaxTile ? h : kSppfMaxTile, tw = w < kSppfMaxTile ? w : kSppfMaxTile;
    const int cg = 32 / (int)sizeof(T);   // two 16-byte vectors of channels per CTA
    const int smem = 2 * (th + 6 * hk) * (tw + 6 * hk) * 32;
    const int tiles_w = (w + tw - 1) / tw, tiles_h = (h + th - 1) / th;
    const dim3 grid(tiles_w * tiles_h, n, (c + cg - 1) / cg);
    if (grid.z > 65535 || n > 65535) return cudaErrorInvalidValue;
    auto launch = [&](auto kern) -> cudaError_t {
        cudaError_t e = set_max_dyn_smem(kern, smem);
        if (e != cudaSuccess) return e;
        return launch_kernel(kern, grid, 256, smem, s, (const T *)x, (T *)y, n, c, h, w, th, tw, tiles_w, nhwc);
    };
    switch (hk) {
    case 0: return launch(sppf_pool_kernel<T, 0>);
    case 1: return launch(sppf_pool_kernel<T, 1>);
    case 2: return launch(sppf_pool_kernel<T, 2>);
    default: return launch(sppf_pool_kernel<T, 3>);
    }
}

cudaError_t launch_sppf_pool(const void *x, void *y, int n, int c, int h, int w, int k, int nhwc, int eb,
                             cudaStream_t s) {
    const int hk = k / 2;   // odd k <= 7 (checked by the caller)
    if (eb == 4) return launch_sppf_typed<float>(x, y, n, c, h, w, hk, nhwc, s);
    if (eb == 2) return launch_sppf_typed<__nv_bfloat16>(x, y, n, c, h, w, hk, nhwc, s);
    return launch_sppf_typed<int8_t>(x, y, n, c, h, w, hk, nhwc, s);
}

cudaError_t launch_dequantize_i8(const int8_t *q, void *out, size_t count, float s, int z, int out_bf16,
                                 cudaStream_t st) {
    const int g = grid_for((count + 15) / 16, 256);
    if (out_bf16) return launch_kernel(dequantize_i8_kernel<__nv_bfloat16>, g, 256, 0, st, q, (__nv_bfloat16 *)out, count, s, z);
    return launch_kernel(dequantize_i8_kernel<float>, g, 256, 0, st, q, (float *)out, count, s, z);
}

cudaError_t launch_quantize_i8(const void *x, int in_bf16, int8_t *q, size_t count, float s, int z, cudaStream_t st) {
    const int g = grid_for((count + 15) / 16, 256);
    if (in_bf16) return launch_kernel(quantize_i8_kernel<__nv_bfloat16>, g, 256, 0, st, (const __nv_bfloat16 *)x, q, count, s, z);
    return launch_kernel(quantize_i8_kernel<float>, g, 256, 0, st, (const float *)x, q, count, s, z);
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
