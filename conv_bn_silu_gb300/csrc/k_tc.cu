// k_tc.cu -- tensor-core variants (TF32, BF16) of the fused Conv2d + folded
// BN + SiLU layer on sm_103a.
//
// Implicit GEMM (page 1, "What NHWC is and why it matters", item 3 and the
// tensor-core plan of "Improvements" #2): the output tile is 128 consecutive
// output pixels (n, oh, ow flattened) x BN output channels.  K is walked as
// (filter tap, channel block); each K step brings
//   A: 128 pixels x RB bytes of channels for one tap, loaded by TMA in im2col
//      mode (the hardware forms the shifted, zero-padded window; no im2col
//      matrix exists in memory), or by a 2-D tiled TMA for 1x1 stride-1
//      layers, where A is the NHWC activation matrix itself;
//   B: BN packed weight rows x RB bytes (2-D tiled TMA);
// into a ring of shared-memory stages guarded by mbarriers.  One thread
// issues tcgen05.mma (M=128, N=BN, accumulator in tensor memory); four
// epilogue warps read the accumulator with tcgen05.ld, add the folded bias,
// apply SiLU and store NHWC or NCHW output at exact addresses.
//
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
// Every mbarrier wait is bounded by wall time; on expiry the kernel records
// a timeout in the library's status word, drains what it issued (again
// bounded), frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "cbs_internal.cuh"
#include "tc_ptx.cuh"

namespace cbs {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kSmemBudget = 200 * 1024;

enum TcKind { kTF32 = 0, kBF16 = 1 };

struct TcParams {
    int M, OH, OW, OHW;
    int C_out;
    int ks, stride, pad;
    int c_in_pad, CB, RB, cblocks, ksteps;
    int BN, stages, a_bytes, b_bytes, stage_bytes;
    int im2col, out_nhwc, out_row_stride;
    uint32_t idesc, swz, tmem_cols;
    const float *bias;
    void *y;
    unsigned int *status;
    // INT8 variant only
    const int32_t *bias_i32;
    const float *m_c;
    float inv_s_y;
    int nchunks, kpc;          // exact-sum K chunks and K steps per chunk
    int stg_bytes;             // int8 staging tile of one stage (128 x CB bytes)
    uint32_t stg_mask;         // staging swizzle mask (bits 7.. -> bits 4..)
    uint32_t op_mask;          // operand swizzle mask
};

__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
tc_conv_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Stage buffers start on a 1024-byte boundary of the shared window (the
    // swizzle atoms of TMA and of the MMA descriptors are address based).
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_addr);
    const int S = p.stages;
    const uint32_t bars = base + S * p.stage_bytes;           // full[S], empty[S], acc_full
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(base_ptr + S * p.stage_bytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_ptr + 2 * S + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    float *bias_s = reinterpret_cast<float *>(tmem_slot + 4);

    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    const uint32_t acc_bar = bars + 8u * (2 * S);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM;
    const int n0 = blockIdx.y * p.BN;
    const int nk = p.ksteps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        ptx::mbar_init(acc_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
        ptx::tmem_relinquish();
    }
    for (int i = threadIdx.x; i < p.BN; i += blockDim.x) {
        const int n = n0 + i;
        bias_s[i] = n < p.C_out ? p.bias[n] : 0.0f;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int issued = 0;  // producer: K steps whose loads were issued
    if (warp == 0) {
        if (lane == 0) {
            // Window corner of the tile's first output pixel.
            const int img = m0 / p.OHW;
            const int rem = m0 - img * p.OHW;
            const int oh = rem / p.OW, ow = rem - (rem / p.OW) * p.OW;
            const int wc = ow * p.stride - p.pad, hc = oh * p.stride - p.pad;
            for (int i = 0; i < nk; ++i) {
                const int s = i % S, u = i / S;
                if (!ptx::mbar_wait_bounded(empty_bar(s), (u & 1) ^ 1, kWaitLimitNs)) {
                    atomicOr(p.status, 1u);
                    *(volatile int *)abort_flag = 1;
                    break;
                }
                if (*(volatile int *)abort_flag) break;
                const int tap = i / p.cblocks, cb = i - tap * p.cblocks;
                const int r = tap / p.ks, t = tap - r * p.ks;
                const uint32_t a_dst = base + s * p.stage_bytes;
                const uint32_t b_dst = a_dst + p.a_bytes;
                ptx::mbar_arrive_expect_tx(full_bar(s), (uint32_t)(p.a_bytes + p.b_bytes));
                if (p.im2col)
                    ptx::tma_load_im2col_4d(a_dst, &tmA, full_bar(s), cb * p.CB, wc, hc, img, (uint16_t)t,
                                            (uint16_t)r);
                else
                    ptx::tma_load_2d(a_dst, &tmA, full_bar(s), cb * p.CB, m0);
                ptx::tma_load_2d(b_dst, &tmB, full_bar(s), tap * p.c_in_pad + cb * p.CB, n0);
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sbo = 8u * p.RB;
            const int kslices = p.RB / 32;
            for (int i = 0; i < nk; ++i) {
                const int s = i % S, u = i / S;
                if (!ptx::mbar_wait_bounded(full_bar(s), u & 1, kWaitLimitNs)) {
                    atomicOr(p.status, 1u);
                    *(volatile int *)abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t a_addr = base + s * p.stage_bytes;
                const uint32_t b_addr = a_addr + p.a_bytes;
                for (int j = 0; j < kslices; ++j) {
                    const uint64_t ad = ptx::smem_desc(a_addr + 32u * j, 16u, sbo, p.swz);
                    const uint64_t bd = ptx::smem_desc(b_addr + 32u * j, 16u, sbo, p.swz);
                    if (KIND == kTF32)
                        ptx::mma_tf32(tmem_base, ad, bd, p.idesc, (i > 0 || j > 0) ? 1u : 0u);
                    else
                        ptx::mma_f16(tmem_base, ad, bd, p.idesc, (i > 0 || j > 0) ? 1u : 0u);
                }
                ptx::mma_commit(empty_bar(s));
            }
            ptx::mma_commit(acc_bar);  // fires once every MMA above has completed
        }
    } else {
        // Epilogue warps 2..5.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const int m = m0 + row;
        const bool ok = ptx::mbar_wait_bounded(acc_bar, 0, kWaitLimitNs);
        if (!ok) {
            atomicOr(p.status, 1u);
            *(volatile int *)abort_flag = 1;
        }
        ptx::tc_fence_after();
        int img = 0, oh = 0, ow = 0;
        if (m < p.M) {
            img = m / p.OHW;
            const int rem = m - img * p.OHW;
            oh = rem / p.OW;
            ow = rem - oh * p.OW;
        }
        const bool valid = ok && m < p.M && !*(volatile int *)abort_flag;
        for (int c0 = 0; c0 < p.BN; c0 += 16) {
            uint32_t v[16];
            ptx::tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
            ptx::tmem_ld_wait();
            if (!valid) continue;
            float o[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = silu_fast(__uint_as_float(v[j]) + bias_s[c0 + j]);
            const int nbase = n0 + c0;
            if (p.out_nhwc) {
                if (KIND == kTF32) {
                    float *yr = static_cast<float *>(p.y) + (size_t)m * p.C_out + nbase;
                    if (nbase + 16 <= p.C_out && (p.C_out & 3) == 0) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(yr + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                    } else {
                        for (int j = 0; j < 16 && nbase + j < p.C_out; ++j) yr[j] = o[j];
                    }
                } else {
                    __nv_bfloat16 *yr = static_cast<__nv_bfloat16 *>(p.y) + (size_t)m * p.C_out + nbase;
                    if (nbase + 16 <= p.C_out && (p.C_out & 7) == 0) {
                        uint32_t w[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * j], o[2 * j + 1]);
                            w[j] = *reinterpret_cast<uint32_t *>(&h2);
                        }
                        *reinterpret_cast<uint4 *>(yr) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4 *>(yr + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {
                        for (int j = 0; j < 16 && nbase + j < p.C_out; ++j) yr[j] = __float2bfloat16_rn(o[j]);
                    }
                }
            } else {
                // NCHW: lanes hold consecutive pixels, so each channel's
                // store is contiguous across the warp.
                const size_t plane = (size_t)p.OH * p.out_row_stride;
                const size_t pix = (size_t)oh * p.out_row_stride + ow;
                for (int j = 0; j < 16; ++j) {
                    const int n = nbase + j;
                    if (n >= p.C_out) break;
                    const size_t off = ((size_t)img * p.C_out + n) * plane + pix;
                    if (KIND == kTF32)
                        static_cast<float *>(p.y)[off] = o[j];
                    else
                        static_cast<__nv_bfloat16 *>(p.y)[off] = __float2bfloat16_rn(o[j]);
                }
            }
        }
    }

    // ---- teardown: all tensor-memory reads done, all copies landed.
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && *(volatile int *)abort_flag) {
        // Drain loads still in flight after an abort (bounded).
        for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
            ptx::mbar_wait_bounded(full_bar(i % S), (i / S) & 1, kWaitLimitNs);
    }
    if (warp == 1 && *(volatile int *)abort_flag && lane == 0) {
        ptx::mbar_wait_bounded(acc_bar, 0, kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------------ INT8
// INT8 layer on the tensor cores.  sm_103a has no integer MMA kind, so int8
// codes are widened to bfloat16, which holds every value in [-128, 127]
// exactly; products (|q_x q_w| <= 16256) are exact, and an FP32 accumulator
// stays exact while |sum| < 2^24, i.e. for at most 1024 products.  The K
// walk is therefore cut into chunks of <= 1024 and each chunk accumulates in
// its own TMEM columns; the epilogue converts every chunk to int32 (exact)
// and sums them in integer arithmetic with the int32 bias.
//
// Pipeline per K step: TMA (int8 activations -> staging, bf16 weights ->
// operand B) -> epilogue warps widen the staging tile into operand A
// (swizzled, then fence.proxy.async) -> one thread issues the MMAs.  The same
// four warps run the requantising epilogue after the last K step.

// Our exp for the requantising epilogue, specified bit for bit:
// Cody-Waite reduction with a 16-bit head of ln 2, degree-7 Taylor
// polynomial in Horner form with fused multiply-adds, scaling by 2^k through
// the exponent field; +inf above 88, +0 below -87.
__device__ __forceinline__ float cw_exp(float x) {
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

// q = rne(clamp(SiLU(float(acc) * m_c) * inv_s_y, -128, 127)), IEEE steps.
__device__ __forceinline__ int requant_i8(int acc, float m_c, float inv_s_y) {
    const float t = __fmul_rn(__int2float_rn(acc), m_c);
    const float e = cw_exp(-t);
    const float u = __fdiv_rn(t, __fadd_rn(1.0f, e));
    float v = __fmul_rn(u, inv_s_y);
    v = fminf(fmaxf(v, -128.0f), 127.0f);
    return (int)rintf(v);
}

// Address swizzle of the TMA/UMMA shared-memory layouts: 16-byte chunk bits
// [4, 4+b) XOR row bits [7, 7+b), b = 1, 2, 3 for 32-, 64-, 128-byte spans.
__device__ __forceinline__ uint32_t swz(uint32_t addr, uint32_t mask) {
    return addr ^ (((addr >> 7) & mask) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t u_lo, uint32_t u_hi) {
    // u = (q + 128) as an unsigned byte; 2^23 + u - (2^23 + 128) = q exactly,
    // and q's float bits end in 16 zero bits, so the high half is its bf16.
    const float lo = __int_as_float(0x4B000000 | u_lo) - 8388736.0f;
    const float hi = __int_as_float(0x4B000000 | u_hi) - 8388736.0f;
    return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kThreads, 1)
tc_conv_i8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_addr);
    const int S = p.stages;
    // Stage s: [operand A bf16 | operand B bf16 | staging A int8], each 1024-aligned.
    const uint32_t bars = base + S * p.stage_bytes;   // raw_full[S], conv_done[S], free[S], acc_full
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(base_ptr + S * p.stage_bytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_ptr + 3 * S + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    int *bias_s = reinterpret_cast<int *>(tmem_slot + 4);
    float *mc_s = reinterpret_cast<float *>(bias_s + p.BN);

    auto raw_bar = [&](int s) { return bars + 8u * s; };
    auto conv_bar = [&](int s) { return bars + 8u * (S + s); };
    auto free_bar = [&](int s) { return bars + 8u * (2 * S + s); };
    const uint32_t acc_bar = bars + 8u * (3 * S);
    const int op_b_off = p.a_bytes;
    const int stg_off = (p.a_bytes + p.b_bytes + 1023) & ~1023;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM;
    const int n0 = blockIdx.y * p.BN;
    const int nk = p.ksteps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(raw_bar(s), 1);
            ptx::mbar_init(conv_bar(s), 4);   // one arrive per converter warp
            ptx::mbar_init(free_bar(s), 1);
        }
        ptx::mbar_init(acc_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
        ptx::tmem_relinquish();
    }
    for (int i = threadIdx.x; i < p.BN; i += blockDim.x) {
        const int n = n0 + i;
        bias_s[i] = n < p.C_out ? p.bias_i32[n] : 0;
        mc_s[i] = n < p.C_out ? p.m_c[n] : 0.0f;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            const int img = m0 / p.OHW;
            const int rem = m0 - img * p.OHW;
            const int oh = rem / p.OW, ow = rem - (rem / p.OW) * p.OW;
            const int wc = ow * p.stride - p.pad, hc = oh * p.stride - p.pad;
            for (int i = 0; i < nk; ++i) {
                const int s = i % S, u = i / S;
                if (!ptx::mbar_wait_bounded(free_bar(s), (u & 1) ^ 1, kWaitLimitNs)) {
                    atomicOr(p.status, 1u);
                    *(volatile int *)abort_flag = 1;
                    break;
                }
                if (*(volatile int *)abort_flag) break;
                const int tap = i / p.cblocks, cb = i - tap * p.cblocks;
                const int r = tap / p.ks, t = tap - r * p.ks;
                const uint32_t st = base + s * p.stage_bytes;
                ptx::mbar_arrive_expect_tx(raw_bar(s), (uint32_t)(p.stg_bytes + p.b_bytes));
                if (p.im2col)
                    ptx::tma_load_im2col_4d(st + stg_off, &tmA, raw_bar(s), cb * p.CB, wc, hc, img, (uint16_t)t,
                                            (uint16_t)r);
                else
                    ptx::tma_load_2d(st + stg_off, &tmA, raw_bar(s), cb * p.CB, m0);
                ptx::tma_load_2d(st + op_b_off, &tmB, raw_bar(s), tap * p.c_in_pad + cb * p.CB, n0);
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sbo = 8u * p.RB;
            const int kslices = p.RB / 32;
            for (int i = 0; i < nk; ++i) {
                const int s = i % S, u = i / S;
                if (!ptx::mbar_wait_bounded(conv_bar(s), u & 1, kWaitLimitNs) ||
                    !ptx::mbar_wait_bounded(raw_bar(s), u & 1, kWaitLimitNs)) {
                    atomicOr(p.status, 1u);
                    *(volatile int *)abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const int chunk = i / p.kpc;
                const bool first_of_chunk = (i % p.kpc) == 0;
                const uint32_t d_tmem = tmem_base + (uint32_t)(chunk * p.BN);
                const uint32_t a_addr = base + s * p.stage_bytes;
                const uint32_t b_addr = a_addr + op_b_off;
                for (int j = 0; j < kslices; ++j) {
                    const uint64_t ad = ptx::smem_desc(a_addr + 32u * j, 16u, sbo, p.swz);
                    const uint64_t bd = ptx::smem_desc(b_addr + 32u * j, 16u, sbo, p.swz);
                    ptx::mma_f16(d_tmem, ad, bd, p.idesc, (first_of_chunk && j == 0) ? 0u : 1u);
                }
                ptx::mma_commit(free_bar(s));
            }
            ptx::mma_commit(acc_bar);
        }
    } else {
        // Warps 2..5: widen int8 staging rows to bf16 operand rows, then the
        // requantising epilogue.  Thread (warp - 2) * 32 + lane owns row
        // `row` of every staging tile.
        const int row = (warp - 2) * 32 + lane;
        const int in_bytes = p.CB;            // int8 bytes per row
        bool ok = true;
        for (int i = 0; i < nk && ok; ++i) {
            const int s = i % S, u = i / S;
            if (!ptx::mbar_wait_bounded(raw_bar(s), u & 1, kWaitLimitNs)) {
                atomicOr(p.status, 1u);
                *(volatile int *)abort_flag = 1;
                ok = false;
                break;
            }
            const uint32_t st = base + s * p.stage_bytes;
            const uint32_t src_row = st + stg_off + row * in_bytes;
            const uint32_t dst_row = st + row * p.RB;
            for (int c = 0; c < in_bytes; c += 16) {
                uint32_t w0, w1, w2, w3;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                             : "r"(swz(src_row + c, p.stg_mask)));
                uint32_t o[8];
                const uint32_t ws[4] = {w0 ^ 0x80808080u, w1 ^ 0x80808080u, w2 ^ 0x80808080u, w3 ^ 0x80808080u};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    o[2 * q] = pack_bf16x2(ws[q] & 0xFF, (ws[q] >> 8) & 0xFF);
                    o[2 * q + 1] = pack_bf16x2((ws[q] >> 16) & 0xFF, ws[q] >> 24);
                }
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz(dst_row + 2 * c, p.op_mask)),
                             "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                             : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz(dst_row + 2 * c + 16, p.op_mask)),
                             "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                             : "memory");
            }
            // Make the generic-proxy writes visible to the tensor cores.
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(conv_bar(s));
        }
        const int q = warp & 3;
        const int erow = 32 * q + lane;       // TMEM lane this thread reads
        const int m = m0 + erow;
        ok = ok && ptx::mbar_wait_bounded(acc_bar, 0, kWaitLimitNs);
        if (!ok) {
            atomicOr(p.status, 1u);
            *(volatile int *)abort_flag = 1;
        }
        ptx::tc_fence_after();
        int img = 0, oh = 0, ow = 0;
        if (m < p.M) {
            img = m / p.OHW;
            const int rem = m - img * p.OHW;
            oh = rem / p.OW;
            ow = rem - oh * p.OW;
        }
        const bool valid = ok && m < p.M && !*(volatile int *)abort_flag;
        for (int c0 = 0; c0 < p.BN; c0 += 16) {
            int acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = bias_s[c0 + j];
            for (int ch = 0; ch < p.nchunks; ++ch) {
                uint32_t v[16];
                ptx::tmem_ld16(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(ch * p.BN + c0), v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] += __float2int_rn(__uint_as_float(v[j]));
            }
            if (!valid) continue;
            int8_t qv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) qv[j] = (int8_t)requant_i8(acc[j], mc_s[c0 + j], p.inv_s_y);
            const int nbase = n0 + c0;
            if (p.out_nhwc) {
                int8_t *yr = static_cast<int8_t *>(p.y) + (size_t)m * p.C_out + nbase;
                if (nbase + 16 <= p.C_out && (p.C_out & 15) == 0) {
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        w[j] = (uint32_t)(uint8_t)qv[4 * j] | ((uint32_t)(uint8_t)qv[4 * j + 1] << 8) |
                               ((uint32_t)(uint8_t)qv[4 * j + 2] << 16) | ((uint32_t)(uint8_t)qv[4 * j + 3] << 24);
                    *reinterpret_cast<uint4 *>(yr) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    for (int j = 0; j < 16 && nbase + j < p.C_out; ++j) yr[j] = qv[j];
                }
            } else {
                const size_t plane = (size_t)p.OH * p.out_row_stride;
                const size_t pix = (size_t)oh * p.out_row_stride + ow;
                for (int j = 0; j < 16; ++j) {
                    const int n = nbase + j;
                    if (n >= p.C_out) break;
                    static_cast<int8_t *>(p.y)[((size_t)img * p.C_out + n) * plane + pix] = qv[j];
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && *(volatile int *)abort_flag) {
        for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
            ptx::mbar_wait_bounded(raw_bar(i % S), (i / S) & 1, kWaitLimitNs);
    }
    if (warp == 1 && *(volatile int *)abort_flag && lane == 0) {
        ptx::mbar_wait_bounded(acc_bar, 0, kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
using EncodeIm2colFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const int *, const int *, cuuint32_t, cuuint32_t,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DriverFns {
    EncodeTiledFn tiled = nullptr;
    EncodeIm2colFn im2col = nullptr;
    bool ok = false;
};

const DriverFns &driver_fns() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        void *p1 = nullptr, *p2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p1, 12000, cudaEnableDefault, &q1) ==
                cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p2, 12000, cudaEnableDefault, &q2) ==
                cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            fns.tiled = reinterpret_cast<EncodeTiledFn>(p1);
            fns.im2col = reinterpret_cast<EncodeIm2colFn>(p2);
            fns.ok = true;
        }
    });
    return fns;
}

CUtensorMapSwizzle swizzle_for(int rb) {
    return rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}
// tcgen05 descriptor swizzle codes: 2 = 128B, 4 = 64B, 6 = 32B.
uint32_t desc_swizzle_code(int rb) { return rb == 128 ? 2u : rb == 64 ? 4u : 6u; }

int round_up(int v, int m) { return (v + m - 1) / m * m; }
int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

int elem_bytes_of(int variant) { return variant == CBS_VARIANT_TC_TF32 ? 4 : 2; }

}  // namespace

// Channels per K step for the INT8 variant (int8 bytes per staging row).
int i8_channel_block(int c_in_pad) { return c_in_pad % 64 == 0 ? 64 : (c_in_pad % 32 == 0 ? 32 : 16); }

cbs_status plan_tc(cbs_plan_t &p) {
    const cbs_layer_desc &d = p.desc;
    const bool i8 = p.variant == CBS_VARIANT_TC_INT8;
    const int eb = i8 ? 1 : elem_bytes_of(p.variant);
    int RB, CB, nchunks = 1;
    if (i8) {
        // int8 codes in memory, widened to bf16 operands in shared memory.
        p.c_in_pad = round_up(d.c_in, 16);
        CB = i8_channel_block(p.c_in_pad);
        RB = 2 * CB;
        const int ksteps = d.k * d.k * (p.c_in_pad / CB);
        nchunks = ceil_div(ksteps, 1024 / CB);
    } else {
        // One K step carries RB bytes of channels (32, 64 or 128: a TMA
        // swizzle span); C_in is padded so a pixel holds a multiple of 32 bytes.
        p.c_in_pad = round_up(d.c_in, 32 / eb);
        const int cbytes = p.c_in_pad * eb;
        RB = (cbytes % 128 == 0) ? 128 : (cbytes % 64 == 0) ? 64 : 32;
        CB = RB / eb;
    }
    p.k_gemm = d.k * d.k * p.c_in_pad;
    p.x_bytes = (size_t)d.n * d.h * d.w * p.c_in_pad * eb;
    p.w_packed_bytes = (size_t)d.c_out * p.k_gemm * (p.variant == CBS_VARIANT_TC_TF32 ? 4 : 2);
    if (d.pad > 127 || (p.oh - 1) * d.stride - d.pad - d.h + 1 < -128 || (p.ow - 1) * d.stride - d.pad - d.w + 1 < -128)
        return fail(CBS_ERR_UNSUPPORTED, "padding outside the im2col corner range");
    const long long M = (long long)d.n * p.oh * p.ow;
    p.m_tiles = ceil_div(M, kBM);
    int BN;
    if (d.force_block_n > 0) {
        BN = d.force_block_n;
        if (BN % 16 || BN < 16 || BN > 256) return fail(CBS_ERR_INVALID_ARG, "block_n %d: 16..256, multiple of 16", BN);
    } else {
        BN = d.c_out <= 256 ? round_up(d.c_out, 16) : 256;
        // Prefer more CTAs when the tile grid cannot fill the SMs.
        while (BN > 32 && (BN % 32) == 0 && (long long)p.m_tiles * ceil_div(d.c_out, BN) < kNumSMs) BN /= 2;
        while (nchunks * BN > 512) BN = round_up(BN / 2, 16);
    }
    if (nchunks * BN > 512)
        return fail(CBS_ERR_UNSUPPORTED, "INT8: %d exact-sum chunks x block_n %d exceed 512 TMEM columns", nchunks, BN);
    if (d.force_split_k > 1) return fail(CBS_ERR_UNSUPPORTED, "split-K not built for the tensor-core path yet");
    p.block_m = kBM;
    p.block_n = BN;
    p.block_k = CB;
    p.n_tiles = ceil_div(d.c_out, BN);
    p.split_k = 1;
    int stage = round_up(kBM * RB + BN * RB, 1024);  // stages stay 1024-byte aligned
    if (i8) stage += round_up(kBM * CB, 1024);       // int8 staging tile
    int stages = kSmemBudget / stage;
    if (stages > 8) stages = 8;
    if (stages < 2) stages = 2;
    p.stages = stages;
    p.threads = kThreads;
    p.smem_bytes = 1024 + stages * stage + 8 * ((i8 ? 3 : 2) * stages + 1) + 16 + BN * (i8 ? 8 : 4);
    p.grid_ctas = p.m_tiles * p.n_tiles;
    p.workspace_bytes = 0;
    return CBS_OK;
}

cbs_status launch_tc(const cbs_plan_t &pl, const void *x, const void *w_packed, const void *bias,
                     const float *m_c, float inv_s_y, void *y, void *workspace, cudaStream_t s) {
    (void)workspace;
    const cbs_layer_desc &d = pl.desc;
    const DriverFns &fns = driver_fns();
    if (!fns.ok) return fail(CBS_ERR_CUDA, "cannot resolve cuTensorMapEncode* from the driver");
    const bool i8 = pl.variant == CBS_VARIANT_TC_INT8;
    if (pl.variant != CBS_VARIANT_TC_TF32 && pl.variant != CBS_VARIANT_TC_BF16 && !i8)
        return fail(CBS_ERR_UNSUPPORTED, "variant %d", pl.variant);
    const int eb_x = i8 ? 1 : elem_bytes_of(pl.variant);          // activation bytes in memory
    const int eb_w = pl.variant == CBS_VARIANT_TC_TF32 ? 4 : 2;   // operand bytes in shared memory
    const CUtensorMapDataType dt_x = pl.variant == CBS_VARIANT_TC_TF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapDataType dt_w = pl.variant == CBS_VARIANT_TC_TF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int CB = pl.block_k;           // channels per K step
    const int RB = CB * eb_w;            // operand row bytes
    const int XB = CB * eb_x;            // activation row bytes as loaded
    const int BN = pl.block_n;

    TcParams P{};
    P.M = d.n * pl.oh * pl.ow;
    P.OH = pl.oh; P.OW = pl.ow; P.OHW = pl.oh * pl.ow;
    P.C_out = d.c_out;
    P.ks = d.k; P.stride = d.stride; P.pad = d.pad;
    P.c_in_pad = pl.c_in_pad; P.CB = CB; P.RB = RB;
    P.cblocks = pl.c_in_pad / CB;
    P.ksteps = d.k * d.k * P.cblocks;
    P.BN = BN; P.stages = pl.stages;
    P.a_bytes = kBM * RB; P.b_bytes = BN * RB;
    P.stage_bytes = round_up(P.a_bytes + P.b_bytes, 1024);
    if (i8) {
        P.stg_bytes = kBM * CB;
        P.stage_bytes += round_up(P.stg_bytes, 1024);
        P.kpc = 1024 / CB;
        P.nchunks = ceil_div(P.ksteps, P.kpc);
        P.stg_mask = XB == 64 ? 3u : XB == 32 ? 1u : 0u;
        P.op_mask = RB == 128 ? 7u : RB == 64 ? 3u : 1u;
        P.bias_i32 = static_cast<const int32_t *>(bias);
        P.m_c = m_c;
        P.inv_s_y = inv_s_y;
    } else {
        P.nchunks = 1;
        P.bias = static_cast<const float *>(bias);
    }
    P.im2col = !(d.k == 1 && d.stride == 1 && d.pad == 0);
    P.out_nhwc = d.out_layout == CBS_NHWC;
    P.out_row_stride = pl.out_row_stride;
    const uint32_t fmt = pl.variant == CBS_VARIANT_TC_TF32 ? 2u : 1u;  // TF32 : BF16 operands
    P.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
    P.swz = desc_swizzle_code(RB);
    const int cols = next_pow2(P.nchunks * BN);
    P.tmem_cols = (uint32_t)(cols < 32 ? 32 : cols);
    P.y = y;
    P.status = device_status_word();
    if (!P.status) return fail(CBS_ERR_CUDA, "cannot resolve the device status word");

    alignas(64) CUtensorMap tmA, tmB;
    CUresult r;
    const cuuint32_t estr1[2] = {1, 1};
    const CUtensorMapSwizzle swz_x = XB == 16 ? CU_TENSOR_MAP_SWIZZLE_NONE : swizzle_for(XB);
    if (P.im2col) {
        const cuuint64_t dims[4] = {(cuuint64_t)pl.c_in_pad, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
        const cuuint64_t strides[3] = {(cuuint64_t)pl.c_in_pad * eb_x, (cuuint64_t)d.w * pl.c_in_pad * eb_x,
                                       (cuuint64_t)d.h * d.w * pl.c_in_pad * eb_x};
        // Bounding box of the window corners: from -pad to (O-1)*stride - pad.
        const int lower[2] = {-d.pad, -d.pad};
        const int upper[2] = {(pl.ow - 1) * d.stride - d.pad - (d.w - 1), (pl.oh - 1) * d.stride - d.pad - (d.h - 1)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)d.stride, (cuuint32_t)d.stride, 1};
        r = fns.im2col(&tmA, dt_x, 4, const_cast<void *>(x), dims, strides, lower, upper, (cuuint32_t)CB, kBM, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz_x, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeIm2col failed (%d)", (int)r);
    } else {
        const cuuint64_t dims[2] = {(cuuint64_t)pl.c_in_pad, (cuuint64_t)P.M};
        const cuuint64_t strides[1] = {(cuuint64_t)pl.c_in_pad * eb_x};
        const cuuint32_t box[2] = {(cuuint32_t)CB, (cuuint32_t)kBM};
        r = fns.tiled(&tmA, dt_x, 2, const_cast<void *>(x), dims, strides, box, estr1, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swz_x, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (A) failed (%d)", (int)r);
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)pl.k_gemm, (cuuint64_t)d.c_out};
        const cuuint64_t strides[1] = {(cuuint64_t)pl.k_gemm * eb_w};
        const cuuint32_t box[2] = {(cuuint32_t)CB, (cuuint32_t)BN};
        r = fns.tiled(&tmB, dt_w, 2, const_cast<void *>(w_packed), dims, strides, box, estr1,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(RB), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (B) failed (%d)", (int)r);
    }

    dim3 grid(pl.m_tiles, pl.n_tiles, 1);
    cudaError_t e;
    if (pl.variant == CBS_VARIANT_TC_TF32) {
        e = cudaFuncSetAttribute(tc_conv_kernel<kTF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
        if (e == cudaSuccess) tc_conv_kernel<kTF32><<<grid, kThreads, pl.smem_bytes, s>>>(tmA, tmB, P);
    } else if (pl.variant == CBS_VARIANT_TC_BF16) {
        e = cudaFuncSetAttribute(tc_conv_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
        if (e == cudaSuccess) tc_conv_kernel<kBF16><<<grid, kThreads, pl.smem_bytes, s>>>(tmA, tmB, P);
    } else {
        e = cudaFuncSetAttribute(tc_conv_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
        if (e == cudaSuccess) tc_conv_i8_kernel<<<grid, kThreads, pl.smem_bytes, s>>>(tmA, tmB, P);
    }
    if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute");
    return cuda_check(cudaGetLastError(), "tensor-core kernel launch");
}

}  // namespace cbs
