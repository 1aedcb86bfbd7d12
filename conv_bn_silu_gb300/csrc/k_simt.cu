// k_simt.cu -- FP32 CUDA-core variant of the fused Conv2d + folded BN + SiLU.
//
// Implicit GEMM (page 1, "What NHWC is and why it matters", item 3):
//   A[m, k] = x[n, oh*S-P+r, ow*S-P+s, ci]   (m = (n, oh, ow), k = (r, s, ci))
//   B[k, co] = w'[co, r, s, ci]               (packed [K][C_out] by cbs_fold_bn)
//   y[m, co] = SiLU(sum_k A[m,k] B[k,co] + b'[co])
// The A tile is gathered straight from x (NCHW or NHWC), zero outside the
// image, into shared memory; nothing is materialised in global memory.  A
// per-CTA table maps each k of the CTA's K range to its input offset and
// filter tap, so the gather costs one table read, a bounds test and a load.
// Each thread accumulates a TM x TN register tile with FP32 fused
// multiply-adds.  The epilogue adds the folded bias and applies SiLU, stages
// the output tile in shared memory and stores it so that consecutive lanes
// write consecutive addresses, each element at its exact address (row pitch
// out_row_stride for NCHW): no store reaches the padding columns of a row or
// the next row (page 1, "Bug fixed: TMA overflow in Conv2dBnSiluTiled").
//
// Split-K (small spatial layers at batch 1): CTAs with blockIdx.z = split
// index write their partial tile to the workspace; the last CTA to arrive on
// the tile's counter sums the partials in split order (deterministic), runs
// the epilogue and puts the counter back to zero.  Nothing waits on another
// CTA, so there is no spin loop.
#include "cbs_internal.cuh"
#include "tc_ptx.cuh"

namespace cbs {
namespace {

// z * sigmoid(z) = z / (1 + e^-z).  Hardware exp2 and fast division: the
// relative error stays near 1e-6 over the output range, far inside the FP32
// path's 1e-5 relative-L2 bar, at a fraction of the instruction count.
__device__ __forceinline__ float silu_f32(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

struct KEntry {
    int off;      // input offset of (r, s, ci) relative to the window corner in x; for a
                  // channel of the second input x_b, ~(its offset in x_b) (offsets are >= 0)
    short r, s;   // filter tap (r = kMaxTap marks k beyond the CTA's range)
};
constexpr short kNoTap = 0x3fff;

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
    constexpr int MAIN_FLOATS = 2 * BK * (BM + BN);
    constexpr int CP = BM + 4;           // NCHW output tile: [BN][BM + 4]
    constexpr int CQ = BN + 4;           // NHWC output tile: [BM][BN + 4]
    constexpr int OUT_FLOATS = NHWC_OUT ? BM * CQ : BN * CP;
    constexpr int TILE_FLOATS = MAIN_FLOATS > OUT_FLOATS ? MAIN_FLOATS : OUT_FLOATS;

    // Dynamic shared memory: [double-buffered A/B tiles | output tile] then
    // the k table.
    extern __shared__ float4 smem4[];
    float *smem = reinterpret_cast<float *>(smem4);
    float (*As)[BK][BM] = reinterpret_cast<float (*)[BK][BM]>(smem);
    float (*Bs)[BK][BN] = reinterpret_cast<float (*)[BK][BN]>(smem + 2 * BK * BM);
    KEntry *ktab = reinterpret_cast<KEntry *>(smem + TILE_FLOATS);
    __shared__ int s_is_last;
    // The next grid may be scheduled now: it waits for this one before it
    // touches global memory.
    ptx::griddep_launch_dependents();

    const int t = threadIdx.x;
    const int tx = t % TX, ty = t / TX;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int kbeg = blockIdx.z * a.k_chunk;
    const int kend = min(a.K, kbeg + a.k_chunk);
    const int klen = kend - kbeg;
    const int klen_pad = (klen + BK - 1) / BK * BK;
    const int OHW = a.OH * a.OW;

    // ---- k table for this CTA's K range
    for (int kl = t; kl < klen_pad; kl += NT) {
        KEntry e;
        if (kl < klen) {
            const int k = kbeg + kl;
            const int tap = k / a.C;
            const int ci = k - tap * a.C;
            const int r = tap / a.KS, s = tap - (tap / a.KS) * a.KS;
            if (ci < a.C_a) {
                e.off = NHWC_IN ? (r * a.W + s) * a.C_a + ci : (ci * a.H + r) * a.W + s;
            } else {   // channel concatenation: the rest come from x_b
                const int cj = ci - a.C_a, cb = a.C - a.C_a;
                e.off = ~(NHWC_IN ? (r * a.W + s) * cb + cj : (cj * a.H + r) * a.W + s);
            }
            e.r = (short)r;
            e.s = (short)s;
        } else {
            e.off = 0;
            e.r = kNoTap;
            e.s = 0;
        }
        ktab[kl] = e;
    }

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
    // Rows (ih) and columns (iw) of the window that lie inside the image,
    // as ranges of the tap index: r in [r_lo, r_hi), s in [s_lo, s_hi).
    const int r_lo = mvalid ? max(0, -ih0) : kNoTap, r_hi = mvalid ? min(a.KS, a.H - ih0) : 0;
    const int s_lo = max(0, -iw0), s_hi = min(a.KS, a.W - iw0);
    const float *__restrict__ xw = a.x + (size_t)img * a.C_a * a.H * a.W +
                                   (NHWC_IN ? ((long long)ih0 * a.W + iw0) * a.C_a : (long long)ih0 * a.W + iw0);
    const int c_b = a.C - a.C_a;
    const float *__restrict__ xw_b =
        a.x_b ? a.x_b + (size_t)img * c_b * a.H * a.W +
                    (NHWC_IN ? ((long long)ih0 * a.W + iw0) * c_b : (long long)ih0 * a.W + iw0)
              : xw;

    float ra[A_PT], rb[B_PT];
    auto load_a = [&](int kl0) {
#pragma unroll
        for (int j = 0; j < A_PT; ++j) {
            const KEntry e = ktab[kl0 + ak0 + j * A_KSTEP];
            float v = 0.0f;
            if (e.r >= r_lo && e.r < r_hi && e.s >= s_lo && e.s < s_hi) v = __ldg(e.off >= 0 ? xw + e.off : xw_b + ~e.off);
            ra[j] = v;
        }
    };
    auto load_b = [&](int kl0) {
#pragma unroll
        for (int j = 0; j < B_PT; ++j) {
            const int idx = t + j * NT;
            float v = 0.0f;
            if (idx < BN * BK) {
                const int kl = kl0 + idx / BN, nl = idx % BN;
                const int n = n0 + nl;
                if (kl < klen && n < a.Cout) v = __ldg(a.w + (size_t)(kbeg + kl) * a.Cout + n);
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

    // The k table and the window above come from the launch parameters only;
    // the previous grid in the stream must be complete before any load.
    ptx::griddep_wait();
    __syncthreads();  // k table ready
    if (klen > 0) {
        load_a(0);
        load_b(0);
        store_smem(0);
    }
    __syncthreads();
    int buf = 0;
    for (int kl = 0; kl < klen; kl += BK) {
        const bool more = kl + BK < klen;
        if (more) {
            load_a(kl + BK);
            load_b(kl + BK);
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
        // The sum runs in split order.  Its loads go out eight splits at a
        // time: one CTA reads every partial of the tile, so a load-add-load
        // chain would pay the L2 latency once per split.
        constexpr int kRedBatch = 8;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int g = 0; g < CG; ++g) {
                const float *src = base + row_of(i) * BN + col_of(g * 4);
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int s0 = 0; s0 < a.split; s0 += kRedBatch) {
                    float4 v[kRedBatch];
#pragma unroll
                    for (int b = 0; b < kRedBatch; ++b)
                        if (s0 + b < a.split)
                            v[b] = __ldcg(reinterpret_cast<const float4 *>(src + (size_t)(s0 + b) * (BM * BN)));
#pragma unroll
                    for (int b = 0; b < kRedBatch; ++b)
                        if (s0 + b < a.split) {
                            sum.x += v[b].x; sum.y += v[b].y; sum.z += v[b].z; sum.w += v[b].w;
                        }
                }
                acc[i][g * 4 + 0] = sum.x; acc[i][g * 4 + 1] = sum.y;
                acc[i][g * 4 + 2] = sum.z; acc[i][g * 4 + 3] = sum.w;
            }
    }

    // ---- epilogue: + folded bias, SiLU into the shared output tile, then
    // coalesced exact-address stores.
    float bvals[TN];
#pragma unroll
    for (int j = 0; j < TN; ++j) {
        const int n = n0 + col_of(j);
        bvals[j] = n < a.Cout ? __ldg(a.bias + n) : 0.0f;
    }
    __syncthreads();  // main-loop tiles are no longer read
    float *Cs = smem;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
#pragma unroll
        for (int g = 0; g < RG; ++g) {
            float v[4];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                const float z = acc[g * 4 + ii][j] + bvals[j];
                v[ii] = a.act == CBS_ACT_IDENTITY ? z : silu_f32(z);
            }
            const int r0 = row_of(g * 4), c = col_of(j);
            if (NHWC_OUT) {
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) Cs[(r0 + ii) * CQ + c] = v[ii];
            } else {
                *reinterpret_cast<float4 *>(&Cs[c * CP + r0]) = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
    }
    __syncthreads();
    if (!NHWC_OUT) {
        const int ml = t % BM;
        const int m = m0 + ml;
        if (m < a.M) {
            const int im = m / OHW;
            const int rem = m - im * OHW;
            const int ohh = rem / a.OW;
            const int oww = rem - ohh * a.OW;
            const size_t pix = ((size_t)im * a.Cout * a.OH + ohh) * (size_t)a.out_row_stride + oww;
            float *yb = a.y + pix;
            const float *rb = a.residual ? a.residual + pix : nullptr;
            const size_t plane = (size_t)a.OH * a.out_row_stride;
            for (int nl = t / BM; nl < BN; nl += NT / BM) {
                const int n = n0 + nl;
                if (n < a.Cout) yb[(size_t)n * plane] = Cs[nl * CP + ml] + (rb ? rb[(size_t)n * plane] : 0.0f);
            }
        }
    } else {
        for (int idx = t; idx < BM * BN; idx += NT) {
            const int ml = idx / BN, nl = idx % BN;
            const int m = m0 + ml, n = n0 + nl;
            if (m < a.M && n < a.Cout) {
                const size_t off = (size_t)m * a.Cout + n;
                a.y[off] = Cs[ml * CQ + nl] + (a.residual ? a.residual[off] : 0.0f);
            }
        }
    }
}

template <int BM, int BN, int TM, int TN, bool IN_NHWC, bool OUT_NHWC>
cudaError_t launch_one(dim3 grid, const SimtLaunch &L, cudaStream_t s) {
    constexpr int NT = (BM / TM) * (BN / TN);
    constexpr int main_floats = 2 * kSimtBK * (BM + BN);
    constexpr int out_floats = OUT_NHWC ? BM * (BN + 4) : BN * (BM + 4);
    constexpr int tile_bytes = 4 * (main_floats > out_floats ? main_floats : out_floats);
    const int kpad = (L.k_chunk + kSimtBK - 1) / kSimtBK * kSimtBK;
    const int bytes = tile_bytes + kpad * (int)sizeof(KEntry);
    auto kern = simt_conv_kernel<BM, BN, TM, TN, kSimtBK, IN_NHWC, OUT_NHWC>;
    if (bytes > 48 * 1024) {
        cudaError_t e = set_max_dyn_smem(kern, bytes);
        if (e != cudaSuccess) return e;
    }
    // A plain launch: measured on GB300, programmatic dependent launch made
    // the batch-1 list 20% slower with these kernels.  Their grids are one
    // partial wave of small CTAs, and CTAs scheduled early pile onto the SMs
    // that have room while the previous kernel runs, instead of spreading
    // over all 152.
    kern<<<grid, NT, bytes, s>>>(L);
    return cudaGetLastError();
}

template <int BM, int BN, int TM, int TN>
cudaError_t launch_cfg(const SimtLaunch &L, cudaStream_t s) {
    dim3 grid(L.m_tiles, L.n_tiles, L.split);
    if (L.in_nhwc && L.out_nhwc) return launch_one<BM, BN, TM, TN, true, true>(grid, L, s);
    if (!L.in_nhwc && !L.out_nhwc) return launch_one<BM, BN, TM, TN, false, false>(grid, L, s);
    if (L.in_nhwc) return launch_one<BM, BN, TM, TN, true, false>(grid, L, s);
    return launch_one<BM, BN, TM, TN, false, true>(grid, L, s);
}

}  // namespace

int simt_smem_bytes(int tile, int k_chunk, int out_nhwc) {
    if (tile < 0 || tile >= kNumSimtTiles) return 0;
    const SimtTile T = kSimtTiles[tile];
    const int main_floats = 2 * kSimtBK * (T.bm + T.bn);
    const int out_floats = out_nhwc ? T.bm * (T.bn + 4) : T.bn * (T.bm + 4);
    const int kpad = (k_chunk + kSimtBK - 1) / kSimtBK * kSimtBK;
    return 4 * (main_floats > out_floats ? main_floats : out_floats) + kpad * (int)sizeof(KEntry);
}

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
