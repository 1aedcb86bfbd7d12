// k_simt.cu -- FP32 CUDA-core variant of the fused Conv2d + folded BN + SiLU.
//
// Implicit GEMM (page 1, "What NHWC is and why it matters", item 3):
//   A[m, k] = x[n, oh*S-P+r, ow*S-P+s, ci]   (m = (n, oh, ow), k = (r, s, ci))
//   B[k, co] = w'[co, r, s, ci]               (packed [K][C_out] by cbs_fold_bn)
//   y[m, co] = SiLU(sum_k A[m,k] B[k,co] + b'[co])
// The A tile is gathered straight from x (NCHW or NHWC), zero outside the
// image, into shared memory; nothing is materialised in global memory.
// Each thread accumulates a TM x TN register tile with FP32 fused
// multiply-adds; the epilogue adds the folded bias and applies SiLU with
// IEEE float operations, then stores each output element at its exact
// address (row pitch out_row_stride for NCHW), so no store can reach the
// padding columns of a row or the next row (page 1, "Bug fixed: TMA overflow
// in Conv2dBnSiluTiled").
//
// Split-K (small spatial layers at batch 1): CTAs with blockIdx.z = split
// index write their partial tile to the workspace; the last CTA to arrive on
// the tile's counter sums the partials in split order (deterministic), runs
// the epilogue and puts the counter back to zero.  Nothing waits on another
// CTA, so there is no spin loop.
#include <cstdio>

#include "cbs_internal.cuh"

namespace cbs {
namespace {

__device__ __forceinline__ float silu_ieee(float z) {
    // z * sigmoid(z) = z / (1 + e^-z); IEEE division and accurate expf.
    return z / (1.0f + expf(-z));
}

template <int BM, int BN, int TM, int TN, int BK, bool NHWC_IN, bool NHWC_OUT>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
simt_conv_kernel(const SimtLaunch a) {
    constexpr int TX = BN / TN;
    constexpr int TY = BM / TM;
    constexpr int NT = TX * TY;
    static_assert(NT % BM == 0, "each thread must own exactly one A row");
    static_assert(TM % 4 == 0 && TN % 4 == 0, "register tiles are float4 groups");
    constexpr int A_PT = BM * BK / NT;   // A elements per thread per K step
    constexpr int A_KSTEP = NT / BM;     // k distance between them
    constexpr int B_PT = (BN * BK + NT - 1) / NT;
    constexpr int RG = TM / 4;           // row groups of 4
    constexpr int CG = TN / 4;           // column groups of 4

    __shared__ __align__(16) float As[2][BK][BM];
    __shared__ __align__(16) float Bs[2][BK][BN];
    __shared__ int s_is_last;

    const int t = threadIdx.x;
    const int tx = t % TX, ty = t / TX;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int kbeg = blockIdx.z * a.k_chunk;
    const int kend = min(a.K, kbeg + a.k_chunk);
    const int OHW = a.OH * a.OW;

    // ---- the A row (output pixel) this thread gathers
    const int am = t % BM;
    const int ak0 = t / BM;
    const int mg = m0 + am;
    const bool mvalid = mg < a.M;
    int img = 0, oh = 0, ow = 0;
    if (mvalid) {
        img = mg / OHW;
        const int rem = mg - img * OHW;
        oh = rem / a.OW;
        ow = rem - oh * a.OW;
    }
    const int ih0 = oh * a.stride - a.pad, iw0 = ow * a.stride - a.pad;
    const float *__restrict__ xb = a.x + (size_t)img * a.C * a.H * a.W;

    // Decode state (ci, r, s) of this thread's k indices, advanced by BK per step.
    int dci[A_PT], dr[A_PT], ds[A_PT];
#pragma unroll
    for (int j = 0; j < A_PT; ++j) {
        const int k = kbeg + ak0 + j * A_KSTEP;
        const int tap = k / a.C;
        dci[j] = k - tap * a.C;
        dr[j] = tap / a.KS;
        ds[j] = tap - dr[j] * a.KS;
    }

    float ra[A_PT], rb[B_PT];
    auto load_a = [&](int kb) {
#pragma unroll
        for (int j = 0; j < A_PT; ++j) {
            const int k = kb + ak0 + j * A_KSTEP;
            float v = 0.0f;
            const int ih = ih0 + dr[j], iw = iw0 + ds[j];
            if (mvalid && k < kend && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W) {
                if (NHWC_IN)
                    v = __ldg(xb + ((size_t)ih * a.W + iw) * a.C + dci[j]);
                else
                    v = __ldg(xb + ((size_t)dci[j] * a.H + ih) * a.W + iw);
            }
            ra[j] = v;
        }
    };
    auto advance_a = [&]() {
#pragma unroll
        for (int j = 0; j < A_PT; ++j) {
            dci[j] += BK;
            while (dci[j] >= a.C) {
                dci[j] -= a.C;
                if (++ds[j] == a.KS) { ds[j] = 0; ++dr[j]; }
            }
        }
    };
    auto load_b = [&](int kb) {
#pragma unroll
        for (int j = 0; j < B_PT; ++j) {
            const int idx = t + j * NT;
            float v = 0.0f;
            if (idx < BN * BK) {
                const int kl = idx / BN, nl = idx - (idx / BN) * BN;
                const int k = kb + kl, n = n0 + nl;
                if (k < kend && n < a.Cout) v = __ldg(a.w + (size_t)k * a.Cout + n);
            }
            rb[j] = v;
        }
    };
    auto store_smem = [&](int buf) {
#pragma unroll
        for (int j = 0; j < A_PT; ++j) As[buf][ak0 + j * A_KSTEP][am] = ra[j];
#pragma unroll
        for (int j = 0; j < B_PT; ++j) {
            const int idx = t + j * NT;
            if (idx < BN * BK) Bs[buf][idx / BN][idx % BN] = rb[j];
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    if (kbeg < kend) {
        load_a(kbeg);
        load_b(kbeg);
        store_smem(0);
    }
    __syncthreads();
    int buf = 0;
    for (int kb = kbeg; kb < kend; kb += BK) {
        const bool more = kb + BK < kend;
        if (more) {
            advance_a();
            load_a(kb + BK);
            load_b(kb + BK);
        }
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float av[TM], bv[TN];
#pragma unroll
            for (int g = 0; g < RG; ++g) {
                const float4 v = *reinterpret_cast<const float4 *>(&As[buf][kk][g * (BM / RG) + ty * 4]);
                av[g * 4 + 0] = v.x; av[g * 4 + 1] = v.y; av[g * 4 + 2] = v.z; av[g * 4 + 3] = v.w;
            }
#pragma unroll
            for (int g = 0; g < CG; ++g) {
                const float4 v = *reinterpret_cast<const float4 *>(&Bs[buf][kk][g * (BN / CG) + tx * 4]);
                bv[g * 4 + 0] = v.x; bv[g * 4 + 1] = v.y; bv[g * 4 + 2] = v.z; bv[g * 4 + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (more) store_smem(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }

    // Row/column of register (i, j) inside the CTA tile.
    auto row_of = [&](int i) { return (i / 4) * (BM / RG) + ty * 4 + (i % 4); };
    auto col_of = [&](int j) { return (j / 4) * (BN / CG) + tx * 4 + (j % 4); };

    if (a.split > 1) {
        const int tile_id = blockIdx.y * a.m_tiles + blockIdx.x;
        float *mine = a.partials + ((size_t)tile_id * a.split + blockIdx.z) * (BM * BN);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int g = 0; g < CG; ++g) {
                const float4 v = make_float4(acc[i][g * 4 + 0], acc[i][g * 4 + 1],
                                             acc[i][g * 4 + 2], acc[i][g * 4 + 3]);
                __stcg(reinterpret_cast<float4 *>(mine + row_of(i) * BN + col_of(g * 4)), v);
            }
        __threadfence();
        __syncthreads();
        if (t == 0) {
            const unsigned prev = atomicAdd(a.counters + tile_id, 1u);
            const int last = prev == (unsigned)(a.split - 1);
            if (last) a.counters[tile_id] = 0u;  // ready for the next launch
            s_is_last = last;
        }
        __syncthreads();
        if (!s_is_last) return;
        __threadfence();
        const float *base = a.partials + (size_t)tile_id * a.split * (BM * BN);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int g = 0; g < CG; ++g) {
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int sidx = 0; sidx < a.split; ++sidx) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                        base + (size_t)sidx * (BM * BN) + row_of(i) * BN + col_of(g * 4)));
                    sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                }
                acc[i][g * 4 + 0] = sum.x; acc[i][g * 4 + 1] = sum.y;
                acc[i][g * 4 + 2] = sum.z; acc[i][g * 4 + 3] = sum.w;
            }
    }

    // ---- epilogue: + folded bias, SiLU, exact-address stores
    float bvals[TN];
#pragma unroll
    for (int j = 0; j < TN; ++j) {
        const int n = n0 + col_of(j);
        bvals[j] = n < a.Cout ? __ldg(a.bias + n) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = m0 + row_of(i);
        if (m >= a.M) continue;
        const int im = m / OHW;
        const int rem = m - im * OHW;
        const int ohh = rem / a.OW;
        const int oww = rem - ohh * a.OW;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = n0 + col_of(j);
            if (n >= a.Cout) continue;
            const float v = silu_ieee(acc[i][j] + bvals[j]);
            size_t off;
            if (NHWC_OUT)
                off = (size_t)m * a.Cout + n;
            else
                off = (((size_t)im * a.Cout + n) * a.OH + ohh) * (size_t)a.out_row_stride + oww;
            a.y[off] = v;
        }
    }
}

template <int BM, int BN, int TM, int TN>
cudaError_t launch_cfg(const SimtLaunch &L, cudaStream_t s) {
    constexpr int NT = (BM / TM) * (BN / TN);
    dim3 grid(L.m_tiles, L.n_tiles, L.split);
    if (L.in_nhwc && L.out_nhwc)
        simt_conv_kernel<BM, BN, TM, TN, kSimtBK, true, true><<<grid, NT, 0, s>>>(L);
    else if (!L.in_nhwc && !L.out_nhwc)
        simt_conv_kernel<BM, BN, TM, TN, kSimtBK, false, false><<<grid, NT, 0, s>>>(L);
    else if (L.in_nhwc)
        simt_conv_kernel<BM, BN, TM, TN, kSimtBK, true, false><<<grid, NT, 0, s>>>(L);
    else
        simt_conv_kernel<BM, BN, TM, TN, kSimtBK, false, true><<<grid, NT, 0, s>>>(L);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const SimtLaunch &L, cudaStream_t s) {
    switch (L.tile) {
        case 0: return launch_cfg<128, 128, 8, 8>(L, s);
        case 1: return launch_cfg<128, 64, 8, 8>(L, s);
        case 2: return launch_cfg<64, 64, 4, 4>(L, s);
        case 3: return launch_cfg<128, 32, 4, 4>(L, s);
        case 4: return launch_cfg<256, 16, 4, 4>(L, s);
        case 5: return launch_cfg<64, 128, 4, 8>(L, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace cbs
