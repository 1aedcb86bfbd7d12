// k_tc.cu -- tensor-core variants (TF32, BF16) of the fused Conv2d + folded
// BN + SiLU layer on sm_103a.
//
// Implicit GEMM (page 1, "What NHWC is and why it matters", item 3 and the
// tensor-core plan of "Improvements" #2): a tile is 128 * mmul consecutive
// output pixels (n, oh, ow flattened) x BN output channels, computed as mmul
// M=128 accumulators side by side in tensor memory.  K is walked as
// (filter tap, channel block); each K step brings
//   A: 128 * mmul pixels x RB bytes of channels for one tap in ONE TMA box,
//      in im2col mode (the hardware forms the shifted, zero-padded window; no
//      im2col matrix exists in memory), or as a 2-D tile for 1x1 stride-1
//      layers, where A is the NHWC activation matrix itself;
//   B: BN packed weight rows x RB bytes (2-D tiled TMA), either with every
//      K step or, when the layer's weight tile fits, once per CTA into a
//      resident region that every tile of the launch reuses;
// into a ring of shared-memory stages guarded by mbarriers; one stage carries
// k_group K steps.  One thread issues tcgen05.mma (M=128, N=BN, accumulators
// in tensor memory); eight epilogue warps read the accumulators with
// tcgen05.ld, add the folded bias, apply SiLU and store NHWC or NCHW output at
// exact addresses.
//
// The shape of the pipeline follows what GB300 measures: a warp issuing TMA
// copies gets about one box through every ~570 cycles whatever its size (up
// to ~75 B/cycle per SM in total), and an MMA costs ~90 cycles whenever its
// operands change (N <= 128), plus a few hundred cycles for each barrier the
// issuing thread waits on.  So the kernel moves few, large boxes (tall A
// tiles, resident B) from several producer warps and waits once per stage of
// several K steps.
//
// Warp roles: warps 0-3 = TMA producers, warp 4 = TMEM allocator + MMA issuer,
// warps 5-12 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
// Every mbarrier wait is bounded by wall time; on expiry the kernel records
// a timeout in the library's status word, drains what it issued (again
// bounded), frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "cbs_internal.cuh"
#include "requant.cuh"
#include "tc_ptx.cuh"

namespace cbs {
namespace {

constexpr int kBM = 128;                         // rows of one MMA (one TMEM lane per pixel)
constexpr int kMaxProducers = 4;                 // warps 0..3
constexpr int kMmaWarp = kMaxProducers;          // warp 4: TMEM, and the MMA issuer of sub-tile 0
constexpr int kMmaWarps = 2;                     // warps 4, 5: one MMA issuer per 128-pixel sub-tile
constexpr int kEpiFirst = kMmaWarp + kMmaWarps;  // warps 6..13: epilogue
constexpr int kEpiWarps = 8;                     // two per TMEM lane quadrant
constexpr int kThreads = 32 * (kEpiFirst + kEpiWarps);        // TF32/BF16: 448
constexpr int kMaxProducersI8 = 2;               // INT8: warps 0..1
constexpr int kMmaWarpI8 = kMaxProducersI8;      // warp 2
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr int kSmemBudget = 222 * 1024;           // stages + resident weights + barriers

enum TcKind { kTF32 = 0, kBF16 = 1 };

struct TcParams {
    int M, OH, OW, OHW;
    int C_out;
    int ks, stride, pad;
    int c_in_pad, CB, RB, cblocks, ksteps;
    int BN, stages, a_bytes, b_bytes, stage_bytes;
    int im2col, out_nhwc, out_row_stride;
    uint32_t idesc, swz, tmem_cols;
    int acc_stride;            // TMEM columns of one accumulator buffer
    int m_tiles, n_tiles;      // tile grid walked by the persistent CTAs
    const float *bias;
    void *y;
    unsigned int *status;
    // INT8 variant only
    const int32_t *bias_i32;
    const float *m_c;
    float inv_s_y;
    int nprod;                 // producer warps in use (divides stages)
    int nchunks, kpc;          // exact-sum K chunks and K steps per chunk
    int chunk_stride;          // TMEM columns between chunk accumulators (power of two)
    int stg_bytes;             // int8 staging tile of one stage (128 x CB bytes)
    uint32_t stg_mask;         // staging swizzle mask (bits 7.. -> bits 4..)
    uint32_t op_mask;          // operand swizzle mask
    // TF32/BF16 tall tiles, grouped K steps, resident weights
    int mmul;                  // 128-pixel sub-tiles per tile (one A box of 128*mmul rows)
    int kg;                    // K steps per stage (divides ksteps)
    int b_res;                 // weights resident for the whole launch
    int bnp;                   // TMEM columns between sub-tile accumulators (power of two >= BN)
    int b_tile_stride;         // bytes between B tiles (1024-aligned)
    int b_region;              // bytes of the resident weight region (0 if none)
    int a_box_bytes;           // one A box: 128 * mmul * RB
    int st_mode;               // 1: NHWC output staged in shared memory and written by TMA stores
    int cbw;                   // columns of one staged store block (128 bytes of output)
    int nblk;                  // staged store blocks per tile row: ceil(BN / cbw)
    int stg_bytes_total;       // bytes of the staging region (8 warps x 4 KB) when st_mode
    int bias_smem;             // 1: the folded bias is copied to shared memory at start
    int bias_half;             // 1: that copy holds b / 2 (SiLU's tanh form takes h = (z + b) / 2 as one FMA)
    int bias_bytes_smem;       // bytes reserved for it
    // Windowed A (stride 1, pad k/2): tiles are runs of padded positions
    // q = oh * Wp + ow' of one image (ow' < Wp = W + 2 pad; columns ow' >= OW
    // are computed and dropped), and one TMA box brings the zero-padded input
    // window of a tile and channel block; tap (r, s) is the window viewed from
    // row r * Wp + s on.
    int win;
    int Wp, tiles_per_img, R_box;
    int SB;                    // weight-ring stages when the weights are streamed (windowed)
    int act;                   // cbs_activation
    const void *residual;      // nullable: added after the activation (y's layout and element type)
    // Channel concatenation: channel blocks 0..ca_blocks-1 come from the first
    // input (tensor map A), the rest from the second (tensor map A2, block
    // cb - ca_blocks).  ca_blocks = cblocks with one input.
    int ca_blocks;
    // INT8 zero points (asymmetric activations).  Outside the image the
    // input is a real zero, code zp_x: the converters write that code for
    // the taps of a pixel's window that leave the image (TMA fills 0), and
    // the fold's bias carries -zp_x * sum(q_w), so every tap contributes
    // (q - zp_x) * q_w.
    int zp_x, zp_y;
    int in_h, in_w;
    // Split-K (TF32/BF16, im2col or 2-D A, streamed weights, direct stores):
    // unit u = tile * split + part covers stages [part * nstage / split,
    // (part + 1) * nstage / split) of its tile.  Each epilogue warp writes
    // its region of the FP32 partial tile, column-major ([part][col][row]),
    // and the warp that arrives last for that region (counters[tile][warp])
    // sums the parts in order and runs the epilogue.
    int split;
    float *partials;           // [tiles][split][tile_m * BN]
    unsigned int *counters;    // [tiles][kEpiWarps], zero between launches
    // Fields of the two kernel modes (last, so that the plain kernel's fields
    // keep their offsets).
    int kpar;                  // 2: a 128-pixel tile's stages are split between the two MMA issuers by
                               //    the parity of the stage count g (with an even ring, each ring slot
                               //    always goes to the same issuer), each into its own accumulator,
                               //    added by the epilogue; else 1
    // Stride-2 window (3x3, pad 1): a tile is a block of tile_h output rows x tile_w
    // output columns (ncol blocks across an image), on a grid of Wp = tile_w + 1
    // positions per row; two boxes per window, plane 0 with the even input
    // rows from the block's first output row oh0 on and plane 1 (at
    // plane1_off) with the odd rows from oh0 - 1; a plane row is read as pairs
    // of pixels (PR = 2 RB bytes per operand row, swizzle swz_a), Wp pairs from
    // pair ow0 - 1 on.
    int s2, PR, plane1_off, tile_w, tile_h, ncol;
    uint32_t swz_a;            // descriptor swizzle code of the window's operand rows
    // 3xTF32 with NCHW input: the converter warps read x (N, c_in, in_h, in_w
    // floats) themselves, or (flat boxes) from one TMA box of raw_bytes per
    // K step, landed over the stage's A tiles.
    const float *x_nchw;
    int c_in;
    int raw_bytes;
};

constexpr int kSplitCounterSlots = 8;   // one per epilogue warp

constexpr int kStageBlockBytes = 4096;            // one warp's staged store block: 32 rows x 128 B

// SiLU(z) = z * sigmoid(z) = h + h * tanh(h) with h = z / 2: one MUFU
// operation per output (tanh.approx, relative error ~2^-11, far below the
// TF32/BF16 tolerances and the bfloat16 output rounding).
__device__ __forceinline__ float silu_fast(float z) {
    const float h = 0.5f * z;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// SiLU(z) = z / (1 + e^-z) with the hardware exp and a fast division:
// relative error near 1e-6, inside the FP32 bar (the 3xTF32 variant).
__device__ __forceinline__ float silu_precise(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Bias + SiLU + store of 16 consecutive output channels of one pixel.
template <bool PRECISE = false>
__device__ __forceinline__ float activate(const TcParams &p, float z) {
    return p.act == CBS_ACT_IDENTITY ? z : (PRECISE ? silu_precise(z) : silu_fast(z));
}

// o = act(v + b) for 16 accumulator values.
template <bool PRECISE = false>
__device__ __forceinline__ void activate16(const TcParams &p, const uint32_t (&v)[16], const float (&bv)[16],
                                           float (&o)[16]) {
    if (p.act == CBS_ACT_IDENTITY) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) o[jj] = __uint_as_float(v[jj]) + bv[jj];
    } else if (PRECISE) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) o[jj] = silu_precise(__uint_as_float(v[jj]) + bv[jj]);
    } else if (p.bias_half) {
        // bv holds b / 2: h = z / 2 in one FMA (halving is exact).
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const float h = fmaf(__uint_as_float(v[jj]), 0.5f, bv[jj]);
            float t;
            asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
            o[jj] = fmaf(h, t, h);
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) o[jj] = silu_fast(__uint_as_float(v[jj]) + bv[jj]);
    }
}

// Adds the residual of 16 consecutive channels nbase.. of one output element
// run (NHWC: pixel m; contiguous), channels past C_out excluded.
template <int KIND>
__device__ __forceinline__ void add_residual16_nhwc(const TcParams &p, int m, int nbase, float (&o)[16]) {
    const size_t off = (size_t)m * p.C_out + nbase;
    if (nbase + 16 <= p.C_out && ((p.C_out & (KIND == kTF32 ? 3 : 7)) == 0)) {
        if (KIND == kTF32) {
            const float4 *r = reinterpret_cast<const float4 *>(static_cast<const float *>(p.residual) + off);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = r[q];
                o[4 * q] += v.x; o[4 * q + 1] += v.y; o[4 * q + 2] += v.z; o[4 * q + 3] += v.w;
            }
        } else {
            const uint4 *r = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.residual) + off);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint4 v = r[q];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[k]);
                    o[8 * q + 2 * k] += __low2float(h2);
                    o[8 * q + 2 * k + 1] += __high2float(h2);
                }
            }
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            if (nbase + jj >= p.C_out) break;
            o[jj] += KIND == kTF32 ? static_cast<const float *>(p.residual)[off + jj]
                                   : __bfloat162float(static_cast<const __nv_bfloat16 *>(p.residual)[off + jj]);
        }
    }
}

// The 16 folded-bias values of channels nbase.. (zero past C_out).
__device__ __forceinline__ void load_bias16(const TcParams &p, const float *bias, int nbase, float (&bv)[16]) {
    if (nbase + 16 <= p.C_out) {
#pragma unroll
        for (int jj = 0; jj < 16; jj += 4) {
            const float4 b4 = *reinterpret_cast<const float4 *>(bias + nbase + jj);
            bv[jj] = b4.x; bv[jj + 1] = b4.y; bv[jj + 2] = b4.z; bv[jj + 3] = b4.w;
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) bv[jj] = nbase + jj < p.C_out ? bias[nbase + jj] : 0.0f;
    }
}

// Bias + SiLU of 16 accumulator columns, written into row `row` of a staged
// store block (32 rows x 128 bytes, 128-byte swizzle: 16-byte chunk j of a
// row sits at chunk j ^ (row % 8)).  c is the block column of the first value.
template <int KIND>
__device__ __forceinline__ void stage16(const TcParams &p, uint32_t blk, int row, int c, const float (&bv)[16],
                                        const uint32_t (&v)[16], int m, int nbase) {
    float o[16];
    activate16(p, v, bv, o);
    if (p.residual && m < p.M) add_residual16_nhwc<KIND>(p, m, nbase, o);
    const uint32_t rbase = blk + (uint32_t)row * 128u;
    if (KIND == kTF32) {
        const int j0 = c >> 2;   // 4 floats per chunk
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t a = rbase + ((uint32_t)((j0 + q) ^ (row & 7)) << 4);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(o[4 * q]), "f"(o[4 * q + 1]),
                         "f"(o[4 * q + 2]), "f"(o[4 * q + 3])
                         : "memory");
        }
    } else {
        const int j0 = c >> 3;   // 8 bf16 per chunk
        uint32_t w[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * jj], o[2 * jj + 1]);
            w[jj] = *reinterpret_cast<uint32_t *>(&h2);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t a = rbase + ((uint32_t)((j0 + q) ^ (row & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[4 * q]), "r"(w[4 * q + 1]),
                         "r"(w[4 * q + 2]), "r"(w[4 * q + 3])
                         : "memory");
        }
    }
}

template <int KIND, bool PRECISE = false>
__device__ __forceinline__ void epi_store16(const TcParams &p, const float *bias, int m, int img, int oh, int ow,
                                            int nbase, const uint32_t (&v)[16]) {
    float bv[16];
    const bool full = nbase + 16 <= p.C_out;
    load_bias16(p, bias, nbase, bv);
    float o[16];
    activate16<PRECISE>(p, v, bv, o);
    if (p.residual) {
        if (p.out_nhwc) {
            add_residual16_nhwc<KIND>(p, m, nbase, o);
        } else {
            const size_t plane = (size_t)p.OH * p.out_row_stride;
            const size_t pix = (size_t)oh * p.out_row_stride + ow;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                if (nbase + jj >= p.C_out) break;
                const size_t off = ((size_t)img * p.C_out + nbase + jj) * plane + pix;
                o[jj] += KIND == kTF32 ? static_cast<const float *>(p.residual)[off]
                                       : __bfloat162float(static_cast<const __nv_bfloat16 *>(p.residual)[off]);
            }
        }
    }
    if (p.out_nhwc) {
        if (KIND == kTF32) {
            float *yr = static_cast<float *>(p.y) + (size_t)m * p.C_out + nbase;
            if (full && (p.C_out & 3) == 0) {
#pragma unroll
                for (int jj = 0; jj < 16; jj += 4)
                    *reinterpret_cast<float4 *>(yr + jj) = make_float4(o[jj], o[jj + 1], o[jj + 2], o[jj + 3]);
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    if (nbase + jj < p.C_out) yr[jj] = o[jj];
            }
        } else {
            __nv_bfloat16 *yr = static_cast<__nv_bfloat16 *>(p.y) + (size_t)m * p.C_out + nbase;
            if (full && (p.C_out & 7) == 0) {
                uint32_t w[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * jj], o[2 * jj + 1]);
                    w[jj] = *reinterpret_cast<uint32_t *>(&h2);
                }
                *reinterpret_cast<uint4 *>(yr) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(yr + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    if (nbase + jj < p.C_out) yr[jj] = __float2bfloat16_rn(o[jj]);
            }
        }
    } else {
        // NCHW: lanes hold consecutive pixels, so each channel's store is
        // contiguous across the warp.
        const size_t plane = (size_t)p.OH * p.out_row_stride;
        const size_t pix = (size_t)oh * p.out_row_stride + ow;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            if (nbase + jj >= p.C_out) continue;
            const size_t off = ((size_t)img * p.C_out + nbase + jj) * plane + pix;
            if (KIND == kTF32)
                static_cast<float *>(p.y)[off] = o[jj];
            else
                static_cast<__nv_bfloat16 *>(p.y)[off] = __float2bfloat16_rn(o[jj]);
        }
    }
}

// Tile t of the persistent walk: M-tile major, N-tile minor, so CTAs that
// run at the same time share A rows through L2.  When the grid is a multiple
// of n_tiles, every tile of a CTA has the same N tile (resident weights).
__device__ __forceinline__ void tile_coords(int t, int n_tiles, int tile_m, int &m0, int &n0, int BN) {
    if (n_tiles == 1) {   // most bandwidth-bound layers: no division per tile
        m0 = t * tile_m;
        n0 = 0;
        return;
    }
    const int mt = t / n_tiles;
    m0 = mt * tile_m;
    n0 = (t - mt * n_tiles) * BN;
}

// Work unit u of a launch: its tile and its range of pipeline stages.
__device__ __forceinline__ void unit_range(int u, int split, int nstage, int &t, int &st0, int &st1) {
    if (split == 1) {
        t = u;
        st0 = 0;
        st1 = nstage;
        return;
    }
    t = u / split;
    const int part = u - t * split;
    st0 = (part * nstage) / split;
    st1 = ((part + 1) * nstage) / split;
}

// The MMAs of one K step for one accumulator: kslices K=16 (bf16) / K=8
// (tf32) slices, 32 bytes apart along both operands' rows.  Descriptors are
// built once per launch (dhi: every field but the start address); a slice
// adds 2 to the start-address field (32 bytes >> 4).  The issuing thread does
// little else between MMAs: the tensor pipe's queue is short, and any slack
// in this thread shows up as idle tensor cycles.
template <int KIND>
__device__ __forceinline__ void issue_kstep(uint32_t d, uint64_t dhi, uint32_t a_addr, uint32_t b_addr, uint32_t idesc,
                                            int kslices, bool first) {
    const uint64_t ad = dhi | (uint64_t)((a_addr & 0x3FFFFu) >> 4);
    const uint64_t bd = dhi | (uint64_t)((b_addr & 0x3FFFFu) >> 4);
    if (kslices == 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (first && k == 0) ? 0u : 1u;
            if (KIND == kTF32)
                ptx::mma_tf32(d, ad + 2u * k, bd + 2u * k, idesc, acc);
            else
                ptx::mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, acc);
        }
    } else {
        for (int k = 0; k < kslices; ++k) {
            const uint32_t acc = (first && k == 0) ? 0u : 1u;
            if (KIND == kTF32)
                ptx::mma_tf32(d, ad + 2u * k, bd + 2u * k, idesc, acc);
            else
                ptx::mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, acc);
        }
    }
}

// The same from ready descriptors (the address field advanced by the caller).
template <int KIND>
__device__ __forceinline__ void issue_kstep_desc(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, int kslices,
                                                 bool first) {
    if (kslices == 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t acc = (first && k == 0) ? 0u : 1u;
            if (KIND == kTF32)
                ptx::mma_tf32(d, ad + 2u * k, bd + 2u * k, idesc, acc);
            else
                ptx::mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, acc);
        }
    } else {
        for (int k = 0; k < kslices; ++k) {
            const uint32_t acc = (first && k == 0) ? 0u : 1u;
            if (KIND == kTF32)
                ptx::mma_tf32(d, ad + 2u * k, bd + 2u * k, idesc, acc);
            else
                ptx::mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, acc);
        }
    }
}

// Loads columns c0 .. c0+15 (and c1 .. c1+15 when `two`) of this warp's TMEM
// lanes.  With the issuer split the tile's sum is spread over two
// accumulators, `half` columns apart, and the halves are added (two waits
// instead of one keep a third 16-column array out of the registers).
__device__ __forceinline__ void tmem_ld_acc(uint32_t t_row, uint32_t c0, uint32_t c1, bool two, bool split2,
                                            uint32_t half, uint32_t (&v0)[16], uint32_t (&v1)[16]) {
    ptx::tmem_ld16(t_row + c0, v0);
    if (two) ptx::tmem_ld16(t_row + c1, v1);
    if (!split2) {
        ptx::tmem_ld_wait();
        return;
    }
    uint32_t w[16];
    ptx::tmem_ld16(t_row + half + c0, w);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v0[i] = __float_as_uint(__uint_as_float(v0[i]) + __uint_as_float(w[i]));
    if (two) {
        ptx::tmem_ld16(t_row + half + c1, w);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v1[i] = __float_as_uint(__uint_as_float(v1[i]) + __uint_as_float(w[i]));
    }
}

__device__ __forceinline__ void abort_now(const TcParams &p, int *abort_flag) {
    atomicOr(p.status, 1u);
    *(volatile int *)abort_flag = 1;
}

__device__ __forceinline__ bool aborted(int *abort_flag) { return *(volatile int *)abort_flag != 0; }

// Kernel modes: the plain kernel; the issuer split (a 128-pixel tile's K
// stages alternate between the two MMA issuers); the stride-2 window.  The
// two rarely used paths are instantiations of their own: as runtime branches
// of one kernel they cost the plain path 2-4% (measured on the BF16 and TF32
// lists at batch 16), the epilogue-bound layers most.
constexpr int kModePlain = 0, kModeIssuerSplit = 1, kModeStride2Window = 2;

// Persistent tensor-core kernel (TF32 / BF16).  Each CTA walks the tiles
// t = blockIdx.x, blockIdx.x + gridDim.x, ...; the producers' stage ring and
// the MMA issuer run ahead across tile boundaries, and the accumulators are
// double-buffered in TMEM so the epilogue of tile j overlaps the MMAs of
// tile j+1.
template <int KIND, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
tc_conv_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmY, const TcParams p) {
    constexpr bool KPAR = MODE == kModeIssuerSplit;     // p.kpar == 2
    constexpr bool S2 = MODE == kModeStride2Window;     // p.win && p.s2
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Buffers start on a 1024-byte boundary of the shared window (the
    // swizzle atoms of TMA and of the MMA descriptors are address based).
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_addr);
    const int S = p.stages;
    // [resident B or weight ring][S stages][store staging][bias][barriers:
    //  full[S], empty[S], acc_full[2], acc_empty[2], drain, b_full,
    //  wring_full[SB], wring_empty[SB]]
    const uint32_t b_base = base;
    const uint32_t stage0 = base + p.b_region;
    const uint32_t stg_base = stage0 + S * p.stage_bytes;
    float *bias_sm = reinterpret_cast<float *>(base_ptr + p.b_region + S * p.stage_bytes + p.stg_bytes_total);
    const uint32_t bars = stg_base + p.stg_bytes_total + p.bias_bytes_smem;
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(base_ptr + p.b_region + S * p.stage_bytes + p.stg_bytes_total +
                                                     p.bias_bytes_smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_ptr + 2 * S + 6 + 2 * p.SB);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    const uint32_t bfull_bar = bars + 8u * (2 * S + 5);
    auto wfull_bar = [&](int b) { return bars + 8u * (2 * S + 6 + b); };
    auto wempty_bar = [&](int b) { return bars + 8u * (2 * S + 6 + p.SB + b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = p.ksteps;
    const int nstage = p.win ? p.cblocks : nk / p.kg;   // stages per tile
    const int tile_m = kBM * p.mmul;
    const int num_tiles = p.m_tiles * p.n_tiles;
    const int num_units = num_tiles * p.split;    // split-K: (tile, K part) units
    const int b_step_bytes = p.BN * p.RB;         // bytes of one B tile as loaded

    // Each 128-pixel sub-tile has its own MMA-issuing thread (lane 0 of warp
    // kMmaWarp + sub-tile): a thread that waits on a barrier once per stage
    // issues an MMA only every ~110-160 cycles, against 48-65 cycles of
    // tensor-pipe time for N <= 128, and two issuers overlap their waits.
    // Every barrier the MMAs release counts one commit per issuer.
    // With kpar = 2 each stage is read by one issuer (the one of its count's
    // parity); otherwise by all mmul issuers.
    const uint32_t n_iss = (uint32_t)(p.mmul * (KPAR ? 2 : 1));
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), (uint32_t)p.mmul);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), n_iss);
            ptx::mbar_init(acce_bar(a), kEpiWarps);   // one arrive per epilogue warp
        }
        ptx::mbar_init(drain_bar, n_iss);
        ptx::mbar_init(bfull_bar, 1);                 // producer warp 0 loads the resident weights
        for (int b = 0; b < p.SB; ++b) {
            ptx::mbar_init(wfull_bar(b), 1);
            ptx::mbar_init(wempty_bar(b), n_iss);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmA);
        if (p.ca_blocks < p.cblocks) ptx::prefetch_tmap(&tmA2);
        ptx::prefetch_tmap(&tmB);
        if (p.st_mode) ptx::prefetch_tmap(&tmY);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // This CTA holds its tensor memory: the next grid may be scheduled.  Then
    // wait for the previous one before touching global memory.
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (p.bias_smem && warp >= kEpiFirst) {
        // Only the epilogue warps read the bias: they copy it and wait for
        // one another (named barrier 1) while the producers already load.
        for (int i = threadIdx.x - 32 * kEpiFirst; i < p.C_out; i += 32 * kEpiWarps)
            bias_sm[i] = p.bias_half ? 0.5f * p.bias[i] : p.bias[i];
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
    }
    const uint32_t tmem_base = *tmem_slot;
    const float *bias = p.bias_smem ? bias_sm : p.bias;

    int last_g = -1;  // producer: last stage (global count) whose loads this warp issued
    int last_w = -1;  // weight-ring lane: last weight load (global count) it issued
    bool b_issued = false;
    // Windowed mode with streamed weights: warp 3 keeps the weight ring full
    // (lane b owns ring slot b) and warps 0..nprod-1 (nprod <= 3) load windows.
    const bool wring = p.win && !p.b_res;
    if (wring && warp == kMaxProducers - 1) {
        if (lane < p.SB) {
            int gw = 0;
            for (int t = blockIdx.x; t < num_tiles && !aborted(abort_flag); t += gridDim.x) {
                const int n0 = (t % p.n_tiles) * p.BN;
                bool ok = true;
                // A ring slot holds one kernel row: the weight tiles of its ks taps.
                const uint32_t slot_bytes = (uint32_t)(p.ks * p.b_tile_stride);
                for (int cb = 0; cb < p.cblocks && ok; ++cb) {
                    for (int r = 0; r < p.ks; ++r, ++gw) {
                        if (gw % p.SB != lane) continue;
                        const int u = gw / p.SB;
                        if (!ptx::mbar_wait_bounded(wempty_bar(lane), (u & 1) ^ 1, kWaitLimitNs) || aborted(abort_flag)) {
                            if (!aborted(abort_flag)) abort_now(p, abort_flag);
                            ok = false;
                            break;
                        }
                        ptx::mbar_arrive_expect_tx(wfull_bar(lane), (uint32_t)(p.ks * b_step_bytes));
                        for (int c = 0; c < p.ks; ++c)
                            ptx::tma_load_2d(b_base + lane * slot_bytes + (uint32_t)(c * p.b_tile_stride), &tmB,
                                             wfull_bar(lane), (r * p.ks + c) * p.c_in_pad + cb * p.CB, n0);
                        last_w = gw;
                    }
                }
                if (!ok) break;
            }
        }
    } else if (warp < kMaxProducers) {
        // A TMA box takes an issuing thread ~570 cycles whatever its size,
        // and lanes issue in parallel: lane l of a producer warp issues box l
        // of the stage (A boxes first, then B boxes).
        const int nbox = p.win ? 1 : p.kg * (p.b_res ? 1 : 2);
        if (warp < p.nprod) {
            if (p.b_res && warp == 0 && blockIdx.x < num_tiles) {
                // This CTA's N tile never changes: load its weight tile once.
                const int n0 = (blockIdx.x % p.n_tiles) * p.BN;
                if (lane == 0) ptx::mbar_arrive_expect_tx(bfull_bar, (uint32_t)(nk * b_step_bytes));
                __syncwarp();
                for (int i = lane; i < nk; i += 32) {
                    const int tap = i / p.cblocks, cb = i - tap * p.cblocks;
                    ptx::tma_load_2d(b_base + i * p.b_tile_stride, &tmB, bfull_bar, tap * p.c_in_pad + cb * p.CB, n0);
                }
                b_issued = true;
            }
            // Producer warp `warp` takes the stages g with g % nprod == warp;
            // nprod divides the stage count, so a stage is always refilled by
            // the same warp and its empty-barrier parity cannot alias.
            int g = 0;
            for (int u = blockIdx.x; u < num_units && !aborted(abort_flag); u += gridDim.x) {
                int t, st0, st1;
                unit_range(u, p.split, nstage, t, st0, st1);
                // Stages g .. g + (st1 - st0) - 1 belong to this unit: a unit
                // none of whose stages is this warp's costs no address math
                // (with one stage per tile, each producer owns every nprod-th tile).
                int own = (warp - g) % p.nprod;
                if (own < 0) own += p.nprod;
                if (own >= st1 - st0) {
                    g += st1 - st0;
                    continue;
                }
                int m0, n0;
                tile_coords(t, p.n_tiles, tile_m, m0, n0, p.BN);
                int img, wc, hc;
                if (S2) {
                    // Stride-2 block: pairs from ow0 - 1, plane rows from oh0 - 1.
                    const int mt = t / p.n_tiles;
                    img = mt / p.tiles_per_img;
                    const int tl = mt - img * p.tiles_per_img;
                    const int rblk = tl / p.ncol;
                    wc = (tl - rblk * p.ncol) * p.tile_w - 1;
                    hc = rblk * p.tile_h - 1;
                } else if (p.win) {
                    // Window of the tile: padded columns -pad .. W+pad-1 of the
                    // input rows from (first output row) - pad on.
                    const int mt = t / p.n_tiles;
                    img = mt / p.tiles_per_img;
                    const int q0 = (mt - img * p.tiles_per_img) * tile_m;
                    wc = -p.pad;
                    hc = q0 / p.Wp - p.pad;
                } else {
                    // Window corner of the tile's first output pixel.
                    img = m0 / p.OHW;
                    const int rem = m0 - img * p.OHW;
                    const int oh = rem / p.OW, ow = rem - (rem / p.OW) * p.OW;
                    wc = ow * p.stride - p.pad;
                    hc = oh * p.stride - p.pad;
                }
                bool ok = true;
                for (int st = st0; st < st1; ++st, ++g) {
                    if (g % p.nprod != warp) continue;
                    const int s = g % S, u = g / S;
                    bool got = true;
                    if (lane == 0) got = ptx::mbar_wait_bounded(empty_bar(s), (u & 1) ^ 1, kWaitLimitNs) && !aborted(abort_flag);
                    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                    if (!got) {
                        if (lane == 0 && !aborted(abort_flag)) abort_now(p, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t sbase = stage0 + s * p.stage_bytes;
                    if (lane == 0)
                        ptx::mbar_arrive_expect_tx(full_bar(s), p.win ? (uint32_t)p.a_box_bytes
                                                                      : (uint32_t)(p.kg * (p.a_box_bytes + (p.b_res ? 0 : b_step_bytes))));
                    __syncwarp();
                    if (S2) {
                        // Stride 2: plane 0 (even input rows) from output row
                        // hc + 1 = oh0 on, plane 1 (odd rows) from oh0 - 1;
                        // both from pair wc = -1 on.
                        if (lane == 0)
                            ptx::tma_load_4d(sbase, &tmA, full_bar(s), 0, wc, hc + 1, img);
                        else if (lane == 1)
                            ptx::tma_load_4d(sbase + (uint32_t)p.plane1_off, &tmA2, full_bar(s), 0, wc, hc, img);
                    } else if (p.win) {
                        // A window stage is channel block st of the first or the second input.
                        const bool second = st >= p.ca_blocks;
                        if (lane == 0)
                            ptx::tma_load_4d(sbase, second ? &tmA2 : &tmA, full_bar(s),
                                             (second ? st - p.ca_blocks : st) * p.CB, wc, hc, img);
                    } else if (lane < nbox) {
                        const bool is_a = lane < p.kg;
                        const int kk = is_a ? lane : lane - p.kg;
                        const int i = st * p.kg + kk;
                        const int tap = i / p.cblocks, cb = i - tap * p.cblocks;
                        if (is_a) {
                            const uint32_t a_dst = sbase + kk * p.a_box_bytes;
                            const int r = tap / p.ks, tt = tap - r * p.ks;
                            const bool second = cb >= p.ca_blocks;   // channel block of the second input
                            const CUtensorMap *tm = second ? &tmA2 : &tmA;
                            const int c0 = (second ? cb - p.ca_blocks : cb) * p.CB;
                            if (p.im2col)
                                ptx::tma_load_im2col_4d(a_dst, tm, full_bar(s), c0, wc, hc, img, (uint16_t)tt,
                                                        (uint16_t)r);
                            else
                                ptx::tma_load_2d(a_dst, tm, full_bar(s), c0, m0);
                        } else {
                            ptx::tma_load_2d(sbase + p.kg * p.a_box_bytes + kk * p.b_tile_stride, &tmB, full_bar(s),
                                             tap * p.c_in_pad + cb * p.CB, n0);
                        }
                    }
                    last_g = g;
                }
                if (!ok) break;
            }
        }
    } else if (warp < kMmaWarp + kMmaWarps) {
        // The sub-tile whose MMAs this warp issues, or with kpar = 2 the
        // parity of the stages it takes.
        const int mi = warp - kMmaWarp;
        if (lane == 0 && mi < p.mmul * (KPAR ? 2 : 1)) {
            const uint32_t sbo = 8u * p.RB;
            const int kslices = p.RB / 32;
            // one 128-row sub-tile of an A box (stride-2 windows: 128 pairs)
            const uint32_t sub_bytes = KPAR ? 0u : (uint32_t)(kBM * (S2 ? p.PR : p.RB));
            const uint64_t dhi = ptx::smem_desc(0u, 16u, sbo, p.swz);
            // Stride-2 windows: operand rows of PR bytes (pairs of pixels).
            const uint64_t dhi_a = S2 ? ptx::smem_desc(0u, 16u, 8u * (uint32_t)p.PR, p.swz_a) : dhi;
            bool ok = true;
            if (p.b_res && blockIdx.x < num_tiles && !ptx::mbar_wait_bounded(bfull_bar, 0, kWaitLimitNs)) {
                abort_now(p, abort_flag);
                ok = false;
            }
            int g = 0, j = 0, gw = 0;
            for (int u = blockIdx.x; ok && u < num_units && !aborted(abort_flag); u += gridDim.x, ++j) {
                int t, st0, st1;
                unit_range(u, p.split, nstage, t, st0, st1);
                const int acc = j & 1, ua = j >> 1;
                if (!ptx::mbar_wait_bounded(acce_bar(acc), (ua & 1) ^ 1, kWaitLimitNs)) {
                    abort_now(p, abort_flag);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.acc_stride + mi * p.bnp);
                if (p.win) {
                    // Row of the window that holds the tile's first position.
                    const int mt = t / p.n_tiles;
                    const int q0 = (mt - (mt / p.tiles_per_img) * p.tiles_per_img) * tile_m;
                    const int row0 = S2 ? 0 : q0 - (q0 / p.Wp) * p.Wp;   // stride-2 blocks start a window row
                    for (int cb = 0; cb < p.cblocks; ++cb, ++g) {
                        const int s = g % S, u = g / S;
                        if (!ptx::mbar_wait_bounded(full_bar(s), u & 1, kWaitLimitNs)) {
                            abort_now(p, abort_flag);
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t window = stage0 + s * p.stage_bytes;
                        if (S2) {
                            // 3x3 stride 2 (one channel block): kernel row r
                            // reads plane 1 (r = 0, 2; one plane row on for
                            // r = 2) or plane 0 (r = 1); column c reads the
                            // second pixel of pair ow - 1 (c = 0), the first of
                            // pair ow (c = 1) or its second (c = 2).
                            const uint32_t abase = window + (uint32_t)row0 * p.PR + mi * sub_bytes;
                            const uint32_t prow = (uint32_t)(p.Wp * p.PR), p1 = (uint32_t)p.plane1_off;
                            const uint32_t pr = (uint32_t)p.PR, rb = (uint32_t)p.RB;
                            const uint32_t roff[3] = {p1, 0u, p1 + prow};
                            const uint32_t coff[3] = {rb, pr, pr + rb};
                            const uint64_t b_col = (uint64_t)(p.b_tile_stride >> 4);
                            for (int r = 0; r < 3; ++r) {
                                uint64_t bd;
                                int ws = 0;
                                if (p.b_res) {
                                    bd = dhi | (uint64_t)(((b_base + (uint32_t)(3 * r * p.b_tile_stride)) & 0x3FFFFu) >> 4);
                                } else {
                                    ws = gw % p.SB;
                                    if (!ptx::mbar_wait_bounded(wfull_bar(ws), (gw / p.SB) & 1, kWaitLimitNs)) {
                                        abort_now(p, abort_flag);
                                        ok = false;
                                        break;
                                    }
                                    ptx::tc_fence_after();
                                    bd = dhi | (uint64_t)(((b_base + (uint32_t)(ws * 3 * p.b_tile_stride)) & 0x3FFFFu) >> 4);
                                }
                                for (int c = 0; c < 3; ++c, bd += b_col) {
                                    const uint64_t ad = dhi_a | (uint64_t)(((abase + roff[r] + coff[c]) & 0x3FFFFu) >> 4);
                                    issue_kstep_desc<KIND>(d_tmem, ad, bd, p.idesc, kslices, r == 0 && c == 0);
                                }
                                if (!p.b_res) {
                                    ptx::mma_commit(wempty_bar(ws));   // the slot is free once these MMAs are done
                                    ++gw;
                                }
                            }
                            if (!ok) break;
                            ptx::mma_commit(empty_bar(s));
                            continue;
                        }
                        if (p.b_res) {
                            // Resident weights: no wait between taps.  The
                            // descriptors advance by constant steps (address
                            // field in 16-byte units): a tap to the right is one
                            // window row on, a tap below is Wp rows on.  A
                            // thread issuing MMAs pays for every scalar
                            // instruction between them.
                            const uint64_t a_first =
                                dhi | (uint64_t)(((window + (uint32_t)row0 * p.RB + mi * sub_bytes) & 0x3FFFFu) >> 4);
                            const uint64_t b_first =
                                dhi | (uint64_t)(((b_base + (uint32_t)(cb * p.b_tile_stride)) & 0x3FFFFu) >> 4);
                            const uint64_t a_col = (uint64_t)(p.RB >> 4), a_row = (uint64_t)((p.Wp * p.RB) >> 4);
                            const uint64_t b_tap = (uint64_t)((p.cblocks * p.b_tile_stride) >> 4);
                            uint64_t ar = a_first, bd = b_first;
                            for (int r = 0; r < p.ks; ++r, ar += a_row) {
                                uint64_t ad = ar;
                                for (int c = 0; c < p.ks; ++c, ad += a_col, bd += b_tap)
                                    issue_kstep_desc<KIND>(d_tmem, ad, bd, p.idesc, kslices, cb == 0 && r == 0 && c == 0);
                            }
                            ptx::mma_commit(empty_bar(s));
                            continue;
                        }
                        // Streamed weights: one wait per kernel row (its ks taps'
                        // weight tiles share a ring slot).
                        const uint64_t a_first =
                            dhi | (uint64_t)(((window + (uint32_t)row0 * p.RB + mi * sub_bytes) & 0x3FFFFu) >> 4);
                        const uint64_t a_col = (uint64_t)(p.RB >> 4), a_row = (uint64_t)((p.Wp * p.RB) >> 4);
                        const uint64_t b_col = (uint64_t)(p.b_tile_stride >> 4);
                        const uint32_t slot_bytes = (uint32_t)(p.ks * p.b_tile_stride);
                        uint64_t ar = a_first;
                        for (int r = 0; r < p.ks; ++r, ar += a_row) {
                            const int ws = gw % p.SB;
                            if (!ptx::mbar_wait_bounded(wfull_bar(ws), (gw / p.SB) & 1, kWaitLimitNs)) {
                                abort_now(p, abort_flag);
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            uint64_t ad = ar;
                            uint64_t bd = dhi | (uint64_t)(((b_base + ws * slot_bytes) & 0x3FFFFu) >> 4);
                            for (int c = 0; c < p.ks; ++c, ad += a_col, bd += b_col)
                                issue_kstep_desc<KIND>(d_tmem, ad, bd, p.idesc, kslices, cb == 0 && r == 0 && c == 0);
                            ptx::mma_commit(wempty_bar(ws));   // the slot is free once these MMAs are done
                            ++gw;
                        }
                        if (!ok) break;
                        ptx::mma_commit(empty_bar(s));
                    }
                    if (!ok) break;
                    ptx::mma_commit(accf_bar(acc));
                    continue;
                }
                bool fresh = true;   // this issuer's accumulator not yet written for this tile
                for (int st = st0; st < st1; ++st, ++g) {
                    // kpar = 2: the stage belongs to the issuer of g's parity.  The
                    // ring depth is even, so slot g % S always goes to the same
                    // issuer, which takes its uses in order: its parity waits
                    // never see a slot two phases behind.
                    if (KPAR && (g & 1) != mi) continue;
                    const int s = g % S, us = g / S;
                    if (!ptx::mbar_wait_bounded(full_bar(s), us & 1, kWaitLimitNs)) {
                        abort_now(p, abort_flag);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sbase = stage0 + s * p.stage_bytes;
                    // K step kk of the stage: A box kk (this issuer's 128-row
                    // half), B tile st * kg + kk (resident) or kk (in the stage).
                    const uint32_t b0 = p.b_res ? b_base + (uint32_t)(st * p.kg * p.b_tile_stride)
                                                : sbase + (uint32_t)(p.kg * p.a_box_bytes);
                    uint64_t ad = dhi | (uint64_t)(((sbase + mi * sub_bytes) & 0x3FFFFu) >> 4);
                    uint64_t bd = dhi | (uint64_t)((b0 & 0x3FFFFu) >> 4);
                    const uint64_t a_step = (uint64_t)(p.a_box_bytes >> 4), b_step = (uint64_t)(p.b_tile_stride >> 4);
                    for (int kk = 0; kk < p.kg; ++kk, ad += a_step, bd += b_step)
                        issue_kstep_desc<KIND>(d_tmem, ad, bd, p.idesc, kslices, (KPAR ? fresh : st == st0) && kk == 0);
                    fresh = false;
                    ptx::mma_commit(empty_bar(s));
                }
                if (!ok) break;
                ptx::mma_commit(accf_bar(acc));  // fires once this tile's MMAs have completed
            }
            ptx::mma_commit(drain_bar);          // fires once every MMA issued here completed
        }
    } else {
        // Epilogue warps: warp w reads TMEM lanes 32*(w%4) .. +31.  With two
        // sub-tiles the two warps of a lane quadrant take one sub-tile each;
        // with one they take alternate 16-column groups.
        const int q = warp & 3;
        const int widx = warp - kEpiFirst;
        const int h = widx >> 2;
        const int sub = p.mmul == 2 ? h : 0;
        const int cstart = p.mmul == 2 ? 0 : 16 * h;
        const int cstep = p.mmul == 2 ? 16 : 32;
        const int row = sub * kBM + 32 * q + lane;
        int j = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++j) {
            int t, st0, st1;
            unit_range(u, p.split, nstage, t, st0, st1);
            const int acc = j & 1, ua = j >> 1;
            // Warp-uniform decision: tcgen05.ld below needs the whole warp.
            bool ok = !aborted(abort_flag) && ptx::mbar_wait_bounded(accf_bar(acc), ua & 1, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !aborted(abort_flag)) abort_now(p, abort_flag);
                break;
            }
            ptx::tc_fence_after();
            int m0, n0;
            tile_coords(t, p.n_tiles, tile_m, m0, n0, p.BN);
            int m = m0 + row;
            int img = 0, oh = 0, ow = 0;
            bool valid;
            if (S2) {
                // Position row = oh' * Wp + ow' of a stride-2 block: keep it
                // when it lies in the block and in the image.
                const int mt = t / p.n_tiles;
                img = mt / p.tiles_per_img;
                const int tl = mt - img * p.tiles_per_img;
                const int rblk = tl / p.ncol;
                const int ohl = row / p.Wp, owl = row - ohl * p.Wp;
                oh = rblk * p.tile_h + ohl;
                ow = (tl - rblk * p.ncol) * p.tile_w + owl;
                valid = ohl < p.tile_h && owl < p.tile_w && oh < p.OH && ow < p.OW;
                m = (img * p.OH + oh) * p.OW + ow;
            } else if (p.win) {
                // Position q of the padded grid: keep it when ow' < OW.
                const int mt = t / p.n_tiles;
                img = mt / p.tiles_per_img;
                const int q = (mt - img * p.tiles_per_img) * tile_m + row;
                oh = q / p.Wp;
                ow = q - oh * p.Wp;
                valid = oh < p.OH && ow < p.OW;
                m = (img * p.OH + oh) * p.OW + ow;
            } else {
                valid = m < p.M;
                if (valid && !p.out_nhwc) {   // NHWC addresses need only m
                    img = m / p.OHW;
                    const int rem = m - img * p.OHW;
                    oh = rem / p.OW;
                    ow = rem - oh * p.OW;
                }
            }
            const uint32_t t_row = tmem_base + (uint32_t)(acc * p.acc_stride + sub * p.bnp) + ((uint32_t)(32 * q) << 16);
            if (p.split > 1) {
                // This warp's region of the partial tile: rows `row`, columns
                // cstart, cstart + cstep, ... (16 each); column-major, so a
                // warp's 32 rows of one column are 128 contiguous bytes.
                const int part = u - t * p.split;
                float *mine = p.partials + ((size_t)t * p.split + part) * (size_t)(tile_m * p.BN);
                for (int c0 = cstart; c0 < p.BN; c0 += cstep) {
                    uint32_t v[16];
                    ptx::tmem_ld16(t_row + (uint32_t)c0, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) __stcg(mine + (size_t)(c0 + jj) * tile_m + row, __uint_as_float(v[jj]));
                }
                // The accumulator has been read: hand it back to the MMA issuer.
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                __threadfence();
                __syncwarp();
                unsigned int prev = 0u;
                unsigned int *counter = p.counters + (size_t)t * kSplitCounterSlots + widx;
                if (lane == 0) prev = atomicAdd(counter, 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev != (unsigned int)(p.split - 1)) continue;
                // Last part of this region: sum the parts in order, then the epilogue.
                if (lane == 0) *counter = 0u;   // ready for the next launch
                __threadfence();
                const float *parts = p.partials + (size_t)t * p.split * (size_t)(tile_m * p.BN);
                for (int c0 = cstart; c0 < p.BN; c0 += cstep) {
                    float sum[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) sum[jj] = 0.0f;
                    for (int k2 = 0; k2 < p.split; ++k2) {
                        const float *src = parts + (size_t)k2 * (tile_m * p.BN) + (size_t)c0 * tile_m + row;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) sum[jj] += __ldcg(src + (size_t)jj * tile_m);
                    }
                    if (valid && n0 + c0 < p.C_out) {
                        uint32_t v[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) v[jj] = __float_as_uint(sum[jj]);
                        epi_store16<KIND>(p, bias, m, img, oh, ow, n0 + c0, v);
                    }
                }
                continue;
            }
            if (p.st_mode) {
                // Staged NHWC store: the warp's 32 pixels x one block of
                // 128 output bytes go to shared memory, then out with one TMA
                // store (coalesced, asynchronous; rows past M and columns
                // past C_out are clipped by the tensor bounds).
                const uint32_t blk = stg_base + (uint32_t)((warp - kEpiFirst) * kStageBlockBytes);
                const int nblk = p.nblk;
                for (int b = p.mmul == 2 ? 0 : h; b < nblk; b += p.mmul == 2 ? 1 : 2) {
                    const int bc0 = b * p.cbw;
                    const int bcols = p.BN - bc0 < p.cbw ? p.BN - bc0 : p.cbw;
                    if (lane == 0) ptx::bulk_wait_read0();   // the block's previous store has read it
                    __syncwarp();
                    for (int c = 0; c < bcols; c += 32) {
                        uint32_t v0[16], v1[16];
                        const bool two = c + 16 < bcols;
                        tmem_ld_acc(t_row, (uint32_t)(bc0 + c), (uint32_t)(bc0 + c + 16), two, KPAR,
                                    (uint32_t)p.bnp, v0, v1);
                        float bv[16];
                        load_bias16(p, bias, n0 + bc0 + c, bv);
                        stage16<KIND>(p, blk, lane, c, bv, v0, m, n0 + bc0 + c);
                        if (two) {
                            load_bias16(p, bias, n0 + bc0 + c + 16, bv);
                            stage16<KIND>(p, blk, lane, c + 16, bv, v1, m, n0 + bc0 + c + 16);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&tmY, blk, n0 + bc0, m0 + sub * kBM + 32 * q);
                        ptx::bulk_commit();
                    }
                }
            } else {
                for (int c0 = cstart; c0 < p.BN; c0 += 2 * cstep) {
                    // Two loads, one wait: 32 columns in flight per thread.
                    uint32_t v0[16], v1[16];
                    const bool two = c0 + cstep < p.BN;
                    tmem_ld_acc(t_row, (uint32_t)c0, (uint32_t)(c0 + cstep), two, KPAR, (uint32_t)p.bnp, v0, v1);
                    if (valid) {
                        if (n0 + c0 < p.C_out) epi_store16<KIND>(p, bias, m, img, oh, ow, n0 + c0, v0);
                        if (two && n0 + c0 + cstep < p.C_out)
                            epi_store16<KIND>(p, bias, m, img, oh, ow, n0 + c0 + cstep, v1);
                    }
                }
            }
            // This accumulator has been read: hand it back to the MMA issuer.
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
        }
        // Staged stores must finish reading shared memory (and land) before
        // the CTA exits.
        if (p.st_mode && lane == 0) ptx::bulk_wait0();
    }

    // ---- teardown: all MMAs complete, loads landed, TMEM freed.
    __syncthreads();
    if (warp < kMaxProducers && lane == 0 && aborted(abort_flag)) {
        // Drain this warp's loads that may still be in flight (bounded).
        for (int g = last_g; g >= 0 && g > last_g - S; g -= p.nprod)
            ptx::mbar_wait_bounded(full_bar(g % S), (g / S) & 1, kWaitLimitNs);
        if (b_issued) ptx::mbar_wait_bounded(bfull_bar, 0, kWaitLimitNs);
    }
    if (warp == kMaxProducers - 1 && lane < p.SB && last_w >= 0 && aborted(abort_flag))
        ptx::mbar_wait_bounded(wfull_bar(lane), (last_w / p.SB) & 1, kWaitLimitNs);
    if (warp == kMmaWarp && lane == 0) {
        if (!ptx::mbar_wait_bounded(drain_bar, 0, kWaitLimitNs)) atomicOr(p.status, 1u);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
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


// What the converter warps of tc_conv_staged_kernel make of the staging tile.
enum StagedKind { kStagedI8 = 0, kStagedX3 = 1 };

// Warp roles of tc_conv_staged_kernel: producers (warps 0-1), the MMA issuer
// (warp 2), kEpi epilogue warps, 4 converter warps.  The INT8 epilogue's
// specified requantisation (about 35 dependent operations per output) bounds
// the INT8 layers, so INT8 runs 16 epilogue warps, each on 8-column groups;
// X3 runs 8 on 16-column groups.  Epilogue warp w reads TMEM lane quadrant
// w % 4, as tcgen05.ld requires.
// How the 3xTF32 kernel's A operand arrives:
//   kX3Nhwc:   NHWC input, TMA im2col or 2-D boxes into the fp32 staging tile;
//   kX3Gather: NCHW input, the converter warps load it from global memory;
//   kX3Flat:   NCHW input of a stride-1 layer with k = 2 pad + 1 (output grid
//              = input grid), batch 1 or whole tiles per image: a channel
//              row of the image is a flat run of H W floats, and the input
//              of filter tap (r, s) at pixel m of a tile is element
//              m + (r - pad) W + (s - pad) of it, except where s - pad takes
//              a column past the row's ends.  One TMA box of kFlatBoxW
//              pixels x CB channels per K step, from the 16-byte aligned
//              element m0 + (r - pad) W - 4, serves the column offsets
//              -pad .. pad of the filter row (the planner takes pad <= 3);
//              rows above and below the image are the box's zero fill, and
//              the converters zero the columns that wrap.  The box lands
//              over the stage's A tail and head tiles, which the converters
//              then overwrite with the split values (one K step per stage:
//              [B head | B tail | A tail | A head]), so a stage is no larger
//              than the gather's.
constexpr int kX3Nhwc = 0, kX3Gather = 1, kX3Flat = 2;
constexpr int kFlatBoxW = 136;   // 128 pixels + 4 either side

template <int SK, int AMODE = kX3Nhwc>
struct StagedLayout {
    static constexpr int kEpi = SK == kStagedI8 ? 16 : 8;
    static constexpr int kEpiFirst = kMmaWarpI8 + 1;
    static constexpr int kConvFirst = kEpiFirst + kEpi;
    // Converter warps: 4, one row of 32 pixels each; the NCHW modes take 8
    // (two per row, each half of the channels): twice the loads in flight.
    static constexpr int kConv = AMODE != kX3Nhwc ? 8 : 4;
    static constexpr int kThreads = 32 * (kConvFirst + kConv);
    static constexpr int kGroup = SK == kStagedI8 ? 8 : 16;   // accumulator columns per TMEM load
};
static_assert(StagedLayout<kStagedX3>::kEpi <= kSplitCounterSlots, "one split-K counter per X3 epilogue warp");
static_assert(StagedLayout<kStagedI8>::kGroup == 8, "the INT8 epilogue loads its bias and scales as two 16-byte pairs");

// X3 sums at most this many K terms into one TMEM accumulator.  The tensor
// cores' accumulation error grows linearly with the number of terms added
// into one accumulator (measured on GB300: relative L2 ~8e-9 per term, so
// 1.5e-5 at K = 2304 against the FP32 bar of 1e-5); consecutive chunks of K
// go to separate accumulators, summed in order in FP32 by the epilogue.
constexpr int kX3ChunkTerms = 384;

// Sum, in order and in FP32, of 16 accumulator columns over the first nch
// K-step chunks (TMEM column offsets chunk_stride apart).
__device__ __forceinline__ void x3_chunk_sum(uint32_t taddr, int nch, int chunk_stride, float (&sum)[16]) {
    uint32_t v[16];
    ptx::tmem_ld16(taddr, v);
    ptx::tmem_ld_wait();
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) sum[jj] = __uint_as_float(v[jj]);
    for (int ch = 1; ch < nch; ++ch) {
        ptx::tmem_ld16(taddr + (uint32_t)(ch * chunk_stride), v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sum[jj] = __fadd_rn(sum[jj], __uint_as_float(v[jj]));
    }
}

// Persistent kernel whose A operand passes through a staging tile and
// converter warps on its way to the tensor cores.  Warps 0-1: TMA producers;
// warp 2: TMEM + MMA issuer; warps 3-10: epilogue; warps 11-14: converters.
//   kStagedI8: int8 codes widened to bf16 operands (exact), exact integer
//              sums in chunks, the specified requantisation.
//   kStagedX3: fp32 activations split into a TF32 head (written back in
//              place, so the tensor cores see it exactly) and the remainder
//              (the tail); the fold splits the weights the same way.  Each K
//              slice runs three kind::tf32 MMAs (tail x head, head x tail,
//              head x head) into one FP32 accumulator, which drops only the
//              tail x tail term: FP32-level accuracy on the tensor cores.
template <int SK, int AMODE>
__global__ void __launch_bounds__(StagedLayout<SK, AMODE>::kThreads, 1)
tc_conv_staged_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                      const __grid_constant__ CUtensorMap tmB, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_addr);
    const int S = p.stages;
    // Stage s holds kg K steps, each block 1024-aligned:
    //   INT8: [kg x operand A bf16 | kg x operand B bf16 | kg x staging A int8];
    //   X3:   [kg x A tail | kg x B head | kg x B tail | kg x staging A fp32,
    //          the A head once converted].
    // Barriers: raw_full[S], conv_done[S], free[S], acc_full[2], acc_empty[2], drain.
    const uint32_t bars = base + S * p.stage_bytes;
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(base_ptr + S * p.stage_bytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_ptr + 3 * S + 5);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    auto raw_bar = [&](int s) { return bars + 8u * s; };
    auto conv_bar = [&](int s) { return bars + 8u * (S + s); };
    auto free_bar = [&](int s) { return bars + 8u * (2 * S + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (3 * S + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (3 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (3 * S + 4);
    const int kg = p.kg;
    constexpr int NB = SK == kStagedX3 ? 2 : 1;                      // weight tiles per K step
    const int op_b_off = kg * p.a_bytes;                              // a_bytes = 128 x RB: 1 KB multiple
    const int stg_off = op_b_off + NB * kg * p.b_tile_stride;
    const int stg_stride = (p.stg_bytes + 1023) & ~1023;
    const int nstage = p.ksteps / kg;

    using L = StagedLayout<SK, AMODE>;
    constexpr bool GATHER = AMODE == kX3Gather, FLAT = AMODE == kX3Flat;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_tiles = p.m_tiles * p.n_tiles;
    const int num_units = num_tiles * p.split;   // X3 split-K: (tile, K part) units; else tiles

    // GATHER (3xTF32, NCHW input): the producers load the weights only; the
    // converter warps read the activations from global memory themselves.
    // FLAT (one K step per stage): the weight tiles first, then the A tail
    // and head tiles, where the producers land the raw NCHW box.
    static_assert(AMODE == kX3Nhwc || SK == kStagedX3, "the NCHW modes are the 3xTF32 kernel's");
    const int b_off = FLAT ? 0 : op_b_off;
    const int flat_tail = NB * p.b_tile_stride, flat_head = flat_tail + p.a_bytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(raw_bar(s), 1);
            ptx::mbar_init(conv_bar(s), L::kConv);   // one arrive per converter warp
            ptx::mbar_init(free_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), L::kEpi);   // one arrive per epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        if (!GATHER) {
            ptx::prefetch_tmap(&tmA);
            if (p.ca_blocks < p.cblocks) ptx::prefetch_tmap(&tmA2);
        }
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == kMmaWarpI8) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), p.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::griddep_launch_dependents();   // after this CTA's TMEM allocation
    ptx::griddep_wait();
    const uint32_t tmem_base = *tmem_slot;

    int last_g = -1;
    if (warp < kMaxProducersI8) {
        // Producer warp `warp` takes the stages g with g % nprod == warp
        // (nprod divides the stage count: one warp per stage, no aliasing).
        // Lane l issues box l of the stage: A boxes (int8 staging) first,
        // then B boxes; TMA issue throughput scales with issuing lanes.
        if (warp < p.nprod) {
            int g = 0;
            for (int uu = blockIdx.x; uu < num_units && !aborted(abort_flag); uu += gridDim.x) {
                int t, st0, st1;
                unit_range(uu, p.split, nstage, t, st0, st1);
                // Skip, without its address math, a unit none of whose stages
                // g .. g + (st1 - st0) - 1 is this warp's.
                int own = (warp - g) % p.nprod;
                if (own < 0) own += p.nprod;
                if (own >= st1 - st0) {
                    g += st1 - st0;
                    continue;
                }
                int m0, n0;
                tile_coords(t, p.n_tiles, kBM, m0, n0, p.BN);
                const int img = m0 / p.OHW;
                const int rem = m0 - img * p.OHW;
                const int oh = rem / p.OW, ow = rem - (rem / p.OW) * p.OW;
                const int wc = ow * p.stride - p.pad, hc = oh * p.stride - p.pad;
                bool ok = true;
                for (int st = st0; st < st1; ++st, ++g) {
                    if (g % p.nprod != warp) continue;
                    const int s = g % S, u = g / S;
                    bool got = true;
                    if (lane == 0) got = ptx::mbar_wait_bounded(free_bar(s), (u & 1) ^ 1, kWaitLimitNs) && !aborted(abort_flag);
                    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                    if (!got) {
                        if (lane == 0 && !aborted(abort_flag)) abort_now(p, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t sb = base + s * p.stage_bytes;
                    if (lane == 0)
                        ptx::mbar_arrive_expect_tx(
                            raw_bar(s), (uint32_t)(kg * ((GATHER ? 0 : FLAT ? p.raw_bytes : p.stg_bytes) + NB * p.b_bytes)));
                    __syncwarp();
                    if (lane < (1 + NB) * kg && !(GATHER && lane < kg)) {   // GATHER: no A boxes
                        // Lanes 0..kg-1: A boxes; then kg B boxes (X3: kg heads, kg tails).
                        const bool is_a = lane < kg;
                        const int kk = is_a ? lane : (lane - kg) % kg;
                        const int tail = is_a ? 0 : (lane - kg) / kg;
                        const int i = st * kg + kk;
                        const int tap = i / p.cblocks, cb = i - tap * p.cblocks;
                        if (FLAT && is_a) {
                            // Filter row r's pixels of this tile: elements x0 + 4 ..
                            // x0 + 131 (+ s - pad) of channel rows y0 .. y0 + CB - 1.
                            const int r = tap / p.ks;
                            const int x0 = (m0 - img * p.OHW) + (r - p.pad) * p.in_w - 4;
                            const int y0 = img * p.c_in + cb * p.CB;
                            if (x0 & 3) {
                                abort_now(p, abort_flag);   // the planner keeps x0 16-byte aligned
                            } else {
                                ptx::tma_load_2d(sb + flat_tail, &tmA, raw_bar(s), x0, y0);
                            }
                        } else if (is_a) {
                            const int r = tap / p.ks, tt = tap - r * p.ks;
                            const uint32_t dst = sb + stg_off + kk * stg_stride;
                            const bool second = cb >= p.ca_blocks;   // channel block of the second input
                            const CUtensorMap *tm = second ? &tmA2 : &tmA;
                            const int c0 = (second ? cb - p.ca_blocks : cb) * p.CB;
                            if (p.im2col)
                                ptx::tma_load_im2col_4d(dst, tm, raw_bar(s), c0, wc, hc, img, (uint16_t)tt,
                                                        (uint16_t)r);
                            else
                                ptx::tma_load_2d(dst, tm, raw_bar(s), c0, m0);
                        } else {
                            // X3 weight tails are rows C_out.. of the packed weights.
                            ptx::tma_load_2d(sb + b_off + (tail * kg + kk) * p.b_tile_stride, &tmB, raw_bar(s),
                                             tap * p.c_in_pad + cb * p.CB, n0 + tail * p.C_out);
                        }
                    }
                    last_g = g;
                }
                if (!ok) break;
            }
        }
    } else if (warp == kMmaWarpI8) {
        if (lane == 0) {
            const uint32_t sbo = 8u * p.RB;
            const int kslices = p.RB / 32;
            const uint64_t dhi = ptx::smem_desc(0u, 16u, sbo, p.swz);
            int g = 0, j = 0;
            for (int uu = blockIdx.x; uu < num_units && !aborted(abort_flag); uu += gridDim.x, ++j) {
                int t, st0, st1;
                unit_range(uu, p.split, nstage, t, st0, st1);
                const int acc = j & 1, ua = j >> 1;
                if (!ptx::mbar_wait_bounded(acce_bar(acc), (ua & 1) ^ 1, kWaitLimitNs)) {
                    abort_now(p, abort_flag);
                    break;
                }
                ptx::tc_fence_after();
                bool ok = true;
                // K step within the current accumulator chunk, and that chunk
                // (counted, not divided: the issuing thread pays for every
                // instruction between its MMAs).  X3 units start at chunk 0.
                int kc = 0, chunk = 0;
                if constexpr (SK != kStagedX3) {
                    chunk = (st0 * kg) / p.kpc;
                    kc = st0 * kg - chunk * p.kpc;
                }
                for (int st = st0; st < st1; ++st, ++g) {
                    const int s = g % S, u = g / S;
                    // conv_done follows raw_full (the converters waited on it),
                    // and raw_full also carries the B tiles.
                    if (!ptx::mbar_wait_bounded(conv_bar(s), u & 1, kWaitLimitNs) ||
                        !ptx::mbar_wait_bounded(raw_bar(s), u & 1, kWaitLimitNs)) {
                        abort_now(p, abort_flag);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sb = base + s * p.stage_bytes;
                    for (int kk = 0; kk < kg; ++kk) {
                        if constexpr (SK == kStagedX3) {
                            if (kc == p.kpc) {   // this unit's next chunk of K steps
                                kc = 0;
                                ++chunk;
                            }
                            const bool first = kc++ == 0;
                            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.acc_stride + chunk * p.chunk_stride);
                            const uint32_t a_head = sb + (FLAT ? flat_head : stg_off + kk * stg_stride);
                            const uint32_t a_tail = sb + (FLAT ? flat_tail : kk * p.a_bytes);
                            const uint32_t b_head = sb + b_off + kk * p.b_tile_stride;
                            const uint32_t b_tail = sb + b_off + (kg + kk) * p.b_tile_stride;
                            issue_kstep<kTF32>(d_tmem, dhi, a_tail, b_head, p.idesc, kslices, first);
                            issue_kstep<kTF32>(d_tmem, dhi, a_head, b_tail, p.idesc, kslices, false);
                            issue_kstep<kTF32>(d_tmem, dhi, a_head, b_head, p.idesc, kslices, false);
                        } else {
                            if (kc == p.kpc) {
                                kc = 0;
                                ++chunk;
                            }
                            const bool first = kc++ == 0;
                            const uint32_t d_tmem =
                                tmem_base + (uint32_t)(acc * p.acc_stride + chunk * p.chunk_stride);
                            issue_kstep<kBF16>(d_tmem, dhi, sb + kk * p.a_bytes, sb + op_b_off + kk * p.b_tile_stride,
                                               p.idesc, kslices, first);
                        }
                    }
                    ptx::mma_commit(free_bar(s));
                }
                if (!ok) break;
                ptx::mma_commit(accf_bar(acc));
            }
            ptx::mma_commit(drain_bar);
        }
    } else if (warp >= L::kConvFirst && GATHER) {
        // Converters, NCHW input: thread (warp - kConvFirst) * 32 + lane owns
        // row `row` (output pixel m0 + row) of every A tile.  For each K step
        // (filter tap, block of CB channels) it loads its pixel's CB input
        // values from global memory (the 32 threads of a warp read 32
        // consecutive output columns of one channel row), zero outside the
        // image, past C_in and past M, and writes the TF32 head (the value
        // with its low 13 mantissa bits cleared) and the exact remainder into
        // the two operand tiles.
        // Warps kConvFirst + w and kConvFirst + 4 + w share rows 32 w ..
        // 32 w + 31: the first takes channels 0 .. CB/2 - 1 of each K step,
        // the second the rest.
        const int row = ((warp - L::kConvFirst) & 3) * 32 + lane;
        const int ch0 = ((warp - L::kConvFirst) >> 2) * (p.CB / 2), chn = p.CB / 2;
        const size_t plane = (size_t)p.in_h * p.in_w;
        int g = 0;
        for (int uu = blockIdx.x; uu < num_units && !aborted(abort_flag); uu += gridDim.x) {
            int t, st0, st1;
            unit_range(uu, p.split, nstage, t, st0, st1);
            int m0, n0;
            tile_coords(t, p.n_tiles, kBM, m0, n0, p.BN);
            const int m = m0 + row;
            const bool mvalid = m < p.M;
            const int img = mvalid ? m / p.OHW : 0;
            const int rem = mvalid ? m - img * p.OHW : 0;
            const int oh = rem / p.OW, ow = rem - (rem / p.OW) * p.OW;
            const int ih0 = oh * p.stride - p.pad, iw0 = ow * p.stride - p.pad;
            const float *ximg = p.x_nchw + (size_t)img * p.c_in * plane;
            // Filter row, column and channel block of the unit's first K step.
            const int i0 = st0 * kg;
            const int tap0 = i0 / p.cblocks;
            int cbk = i0 - tap0 * p.cblocks, r = tap0 / p.ks, cc = tap0 - (tap0 / p.ks) * p.ks;
            bool ok = true;
            for (int st = st0; st < st1; ++st, ++g) {
                const int s = g % S, u = g / S;
                // The stage's A tiles are free once the MMAs that read them
                // have completed (the producer waits on the same barrier).
                // Warp-uniform: the stage ends in __syncwarp.
                const bool got = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(free_bar(s), (u & 1) ^ 1, kWaitLimitNs));
                if (!got) {
                    if (lane == 0) abort_now(p, abort_flag);
                    ok = false;
                    break;
                }
                const uint32_t sb = base + s * p.stage_bytes;
                for (int kk = 0; kk < kg; ++kk) {
                    const int ih = ih0 + r, iw = iw0 + cc, c0 = cbk * p.CB + ch0;
                    const bool in = mvalid && (unsigned)ih < (unsigned)p.in_h && (unsigned)iw < (unsigned)p.in_w;
                    const float *src = ximg + (in ? (size_t)c0 * plane + (size_t)ih * p.in_w + iw : 0);
                    float v[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        v[c] = (in && c < chn && c0 + c < p.c_in) ? __ldg(src + (size_t)c * plane) : 0.0f;
                    // This warp's channels start ch0 channels (4 ch0 bytes) into the row.
                    const uint32_t head_row = sb + stg_off + kk * stg_stride + row * p.RB + 4 * ch0;
                    const uint32_t tail_row = sb + kk * p.a_bytes + row * p.RB + 4 * ch0;
#pragma unroll
                    for (int c = 0; c < 16; c += 4) {
                        if (c < chn) {
                            uint32_t h[4];
                            float l[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                h[q] = __float_as_uint(v[c + q]) & 0xFFFFE000u;
                                l[q] = __fsub_rn(v[c + q], __uint_as_float(h[q]));
                            }
                            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz(head_row + 4 * c, p.op_mask)),
                                         "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                                         : "memory");
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(swz(tail_row + 4 * c, p.op_mask)),
                                         "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3])
                                         : "memory");
                        }
                    }
                    // The next K step: channel block, then filter column, then row.
                    if (++cbk == p.cblocks) {
                        cbk = 0;
                        if (++cc == p.ks) {
                            cc = 0;
                            ++r;
                        }
                    }
                }
                // Make the generic-proxy writes visible to the tensor cores.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(conv_bar(s));
            }
            if (!ok) break;
        }
    } else if (warp >= L::kConvFirst && FLAT) {
        // Converters, NCHW input in flat boxes (one K step per stage): thread
        // (warp - kConvFirst) * 32 + lane owns row `row` (output pixel m0 +
        // row) of the A tiles, as in the gather above, but reads its values
        // from the stage's raw box (channel c of the K step at element
        // c * kFlatBoxW + row + 4 + s - pad: consecutive rows at consecutive
        // words), zero where the filter column leaves the image row, past
        // C_in and past M.  The box lies over the A tiles, so the eight warps
        // all finish reading before any writes: named barrier 2, whose OR of
        // the warps' failures also makes them leave together.
        const int row = ((warp - L::kConvFirst) & 3) * 32 + lane;
        const int ch0 = ((warp - L::kConvFirst) >> 2) * (p.CB / 2), chn = p.CB / 2;
        int g = 0;
        bool stop = false;
        for (int uu = blockIdx.x; uu < num_units && !stop; uu += gridDim.x) {
            int t, st0, st1;
            unit_range(uu, p.split, nstage, t, st0, st1);
            int m0, n0;
            tile_coords(t, p.n_tiles, kBM, m0, n0, p.BN);
            const int m = m0 + row;
            const bool mvalid = m < p.M;
            const int ow = mvalid ? (m % p.OHW) % p.OW : 0;
            const int tap0 = st0 / p.cblocks;
            int cbk = st0 - tap0 * p.cblocks, cc = tap0 - (tap0 / p.ks) * p.ks;
            for (int st = st0; st < st1; ++st, ++g) {
                const int s = g % S, u = g / S;
                // The raw box and the B tiles have landed; the producer
                // waited for the stage's previous MMAs before loading them.
                const bool got = ptx::mbar_wait_bounded(raw_bar(s), u & 1, kWaitLimitNs);
                const uint32_t sb = base + s * p.stage_bytes;
                const int iw = ow + cc - p.pad, c0 = cbk * p.CB + ch0;
                const bool in = got && mvalid && (unsigned)iw < (unsigned)p.in_w;
                const uint32_t src = sb + flat_tail + 4u * (ch0 * kFlatBoxW + row + 4 + cc - p.pad);
                float v[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    v[c] = 0.0f;
                    if (in && c < chn && c0 + c < p.c_in)
                        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[c]) : "r"(src + 4u * c * kFlatBoxW));
                }
                if (ptx::bar_red_or(2, 32 * L::kConv, !got || aborted(abort_flag))) {
                    if (!got) abort_now(p, abort_flag);
                    stop = true;
                    break;
                }
                const uint32_t head_row = sb + flat_head + row * p.RB + 4 * ch0;
                const uint32_t tail_row = sb + flat_tail + row * p.RB + 4 * ch0;
#pragma unroll
                for (int c = 0; c < 16; c += 4) {
                    if (c < chn) {
                        uint32_t h[4];
                        float l[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            h[q] = __float_as_uint(v[c + q]) & 0xFFFFE000u;
                            l[q] = __fsub_rn(v[c + q], __uint_as_float(h[q]));
                        }
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz(head_row + 4 * c, p.op_mask)),
                                     "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                                     : "memory");
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(swz(tail_row + 4 * c, p.op_mask)),
                                     "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3])
                                     : "memory");
                    }
                }
                // The next K step: channel block, then filter column (the
                // row is the producer's).
                if (++cbk == p.cblocks) {
                    cbk = 0;
                    if (++cc == p.ks) cc = 0;
                }
                // Make the generic-proxy writes visible to the tensor cores.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(conv_bar(s));
            }
        }
    } else if (warp >= L::kConvFirst && SK == kStagedX3) {
        // Converters: thread (warp - kConvFirst) * 32 + lane splits row `row`
        // of every staging tile: head = the value with its low 13 mantissa
        // bits cleared (a TF32 number), tail = value - head (exact).
        const int row = (warp - L::kConvFirst) * 32 + lane;
        int g = 0;
        for (int uu = blockIdx.x; uu < num_units && !aborted(abort_flag); uu += gridDim.x) {
            int t, st0, st1;
            unit_range(uu, p.split, nstage, t, st0, st1);
            bool ok = true;
            for (int st = st0; st < st1; ++st, ++g) {
                const int s = g % S, u = g / S;
                if (!ptx::mbar_wait_bounded(raw_bar(s), u & 1, kWaitLimitNs)) {
                    abort_now(p, abort_flag);
                    ok = false;
                    break;
                }
                const uint32_t sb = base + s * p.stage_bytes;
                for (int kk = 0; kk < kg; ++kk) {
                    const uint32_t head_row = sb + stg_off + kk * stg_stride + row * p.RB;
                    const uint32_t tail_row = sb + kk * p.a_bytes + row * p.RB;
                    for (int c = 0; c < p.RB; c += 16) {
                        const uint32_t ha = swz(head_row + c, p.op_mask);
                        uint32_t w[4];
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                     : "r"(ha));
                        uint32_t h[4];
                        float l[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            h[q] = w[q] & 0xFFFFE000u;
                            l[q] = __fsub_rn(__uint_as_float(w[q]), __uint_as_float(h[q]));
                        }
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ha), "r"(h[0]), "r"(h[1]),
                                     "r"(h[2]), "r"(h[3])
                                     : "memory");
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(swz(tail_row + c, p.op_mask)),
                                     "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3])
                                     : "memory");
                    }
                }
                // Make the generic-proxy writes visible to the tensor cores.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(conv_bar(s));
            }
            if (!ok) break;
        }
    } else if (warp >= L::kConvFirst) {
        // Converters: thread (warp - kConvFirst) * 32 + lane widens row `row`
        // of every staging tile into the swizzled bf16 operand.
        const int row = (warp - L::kConvFirst) * 32 + lane;
        const int in_bytes = p.CB;
        // With an input zero point: the code of a real zero, as a bf16 pair.
        const uint32_t zcode = p.zp_x ? pack_bf16x2((uint32_t)(p.zp_x + 128), (uint32_t)(p.zp_x + 128)) : 0u;
        int g = 0;
        for (int t = blockIdx.x; t < num_tiles && !aborted(abort_flag); t += gridDim.x) {
            bool ok = true;
            // With a zero point: bit tap of `oob` marks a tap of this row's
            // pixel window outside the image (k <= 5: at most 25 taps; larger
            // filters test each tap as it comes).
            int ih0 = 0, iw0 = 0;
            uint32_t oob = 0u;
            if (p.zp_x) {
                int m0, n0;
                tile_coords(t, p.n_tiles, kBM, m0, n0, p.BN);
                const int m = m0 + row < p.M ? m0 + row : m0;
                const int img = m / p.OHW;
                const int rem = m - img * p.OHW;
                const int oh = rem / p.OW;
                ih0 = oh * p.stride - p.pad;
                iw0 = (rem - oh * p.OW) * p.stride - p.pad;
                if (p.ks <= 5)
                    for (int r = 0; r < p.ks; ++r)
                        for (int c2 = 0; c2 < p.ks; ++c2)
                            if ((unsigned)(ih0 + r) >= (unsigned)p.in_h || (unsigned)(iw0 + c2) >= (unsigned)p.in_w)
                                oob |= 1u << (r * p.ks + c2);
            }
            int tap = 0, cbk = 0;   // tap and channel block of the next K step
            for (int st = 0; st < nstage; ++st, ++g) {
                const int s = g % S, u = g / S;
                if (!ptx::mbar_wait_bounded(raw_bar(s), u & 1, kWaitLimitNs)) {
                    abort_now(p, abort_flag);
                    ok = false;
                    break;
                }
                const uint32_t sb = base + s * p.stage_bytes;
                for (int kk = 0; kk < kg; ++kk) {
                const uint32_t src_row = sb + stg_off + kk * stg_stride + row * in_bytes;
                const uint32_t dst_row = sb + kk * p.a_bytes + row * p.RB;
                const int ktap = tap;
                if (++cbk == p.cblocks) {
                    cbk = 0;
                    ++tap;
                }
                if (p.zp_x) {
                    bool out;
                    if (p.ks <= 5) {
                        out = (oob >> ktap) & 1u;
                    } else {
                        const int r = ktap / p.ks, c2 = ktap - r * p.ks;
                        out = (unsigned)(ih0 + r) >= (unsigned)p.in_h || (unsigned)(iw0 + c2) >= (unsigned)p.in_w;
                    }
                    if (out) {
                        // A tap outside the image: every channel is the code of zero.
                        for (int c = 0; c < in_bytes; c += 8)
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(swz(dst_row + 2 * c, p.op_mask)),
                                         "r"(zcode)
                                         : "memory");
                        continue;
                    }
                }
                for (int c = 0; c < in_bytes; c += 16) {
                    uint32_t w0, w1, w2, w3;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                                 : "r"(swz(src_row + c, p.stg_mask)));
                    uint32_t o[8];
                    const uint32_t ws[4] = {w0 ^ 0x80808080u, w1 ^ 0x80808080u, w2 ^ 0x80808080u, w3 ^ 0x80808080u};
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        o[2 * qq] = pack_bf16x2(ws[qq] & 0xFF, (ws[qq] >> 8) & 0xFF);
                        o[2 * qq + 1] = pack_bf16x2((ws[qq] >> 16) & 0xFF, ws[qq] >> 24);
                    }
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz(dst_row + 2 * c, p.op_mask)),
                                 "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(swz(dst_row + 2 * c + 16, p.op_mask)),
                                 "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                                 : "memory");
                }
                }
                // Make the generic-proxy writes visible to the tensor cores.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(conv_bar(s));
            }
            if (!ok) break;
        }
    } else {
        // Epilogue warps: quadrant warp % 4; the kEpi / 4 warps of a quadrant
        // take every (kEpi / 4)-th group of kGroup columns.
        constexpr int G = L::kGroup, NSUB = L::kEpi / 4;
        const int q = warp & 3;
        const int sub = (warp - L::kEpiFirst) >> 2;
        const int erow = 32 * q + lane;
        int j = 0;
        for (int uu = blockIdx.x; uu < num_units; uu += gridDim.x, ++j) {
            int t, st0, st1;
            unit_range(uu, p.split, nstage, t, st0, st1);
            const int acc = j & 1, ua = j >> 1;
            bool ok = !aborted(abort_flag) && ptx::mbar_wait_bounded(accf_bar(acc), ua & 1, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0 && !aborted(abort_flag)) abort_now(p, abort_flag);
                break;
            }
            ptx::tc_fence_after();
            int m0, n0;
            tile_coords(t, p.n_tiles, kBM, m0, n0, p.BN);
            const int m = m0 + erow;
            int img = 0, oh = 0, ow = 0;
            if (m < p.M && !p.out_nhwc) {   // NHWC addresses need only m
                img = m / p.OHW;
                const int rem = m - img * p.OHW;
                oh = rem / p.OW;
                ow = rem - oh * p.OW;
            }
            const uint32_t t_row = tmem_base + (uint32_t)(acc * p.acc_stride) + ((uint32_t)(32 * q) << 16);
            if constexpr (SK == kStagedX3) {
                // K-step chunks this unit wrote (parts of a split differ by a stage).
                const int nch = ((st1 - st0) * kg + p.kpc - 1) / p.kpc;
                if (p.split > 1) {
                    // This warp's region of the partial tile (rows erow,
                    // its column groups), column-major: a warp's 32 rows of
                    // one column are 128 contiguous bytes.
                    const int part = uu - t * p.split;
                    float *mine = p.partials + ((size_t)t * p.split + part) * (size_t)(kBM * p.BN);
                    for (int c0 = G * sub; c0 < p.BN; c0 += G * NSUB) {
                        float sum[16];
                        x3_chunk_sum(t_row + (uint32_t)c0, nch, p.chunk_stride, sum);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) __stcg(mine + (size_t)(c0 + jj) * kBM + erow, sum[jj]);
                    }
                    // The accumulator has been read: hand it back to the MMA issuer.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
                    __threadfence();
                    __syncwarp();
                    unsigned int prev = 0u;
                    unsigned int *counter = p.counters + (size_t)t * kSplitCounterSlots + (warp - L::kEpiFirst);
                    if (lane == 0) prev = atomicAdd(counter, 1u);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    if (prev != (unsigned int)(p.split - 1)) continue;
                    // Last part of this region: sum the parts in order, then the epilogue.
                    if (lane == 0) *counter = 0u;   // ready for the next launch
                    __threadfence();
                    const float *parts = p.partials + (size_t)t * p.split * (size_t)(kBM * p.BN);
                    for (int c0 = G * sub; c0 < p.BN; c0 += G * NSUB) {
                        float sum[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) sum[jj] = 0.0f;
                        for (int k2 = 0; k2 < p.split; ++k2) {
                            const float *src = parts + (size_t)k2 * (kBM * p.BN) + (size_t)c0 * kBM + erow;
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) sum[jj] += __ldcg(src + (size_t)jj * kBM);
                        }
                        if (m < p.M && n0 + c0 < p.C_out) {
                            uint32_t v[16];
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) v[jj] = __float_as_uint(sum[jj]);
                            epi_store16<kTF32, true>(p, p.bias, m, img, oh, ow, n0 + c0, v);
                        }
                    }
                    continue;
                }
                for (int c0 = G * sub; c0 < p.BN; c0 += G * NSUB) {
                    float sum[16];
                    x3_chunk_sum(t_row + (uint32_t)c0, nch, p.chunk_stride, sum);
                    if (m >= p.M || n0 + c0 >= p.C_out) continue;
                    uint32_t v[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = __float_as_uint(sum[jj]);
                    epi_store16<kTF32, true>(p, p.bias, m, img, oh, ow, n0 + c0, v);
                }
            } else {
                for (int c0 = G * sub; c0 < p.BN; c0 += G * NSUB) {
                    const int nbase = n0 + c0;
                    int accv[G];
                    float mcv[G];
                    if (nbase + G <= p.C_out) {   // G = 8: two 16-byte loads each (both arrays 16-byte aligned)
                        const int4 b0 = __ldg(reinterpret_cast<const int4 *>(p.bias_i32 + nbase));
                        const int4 b1 = __ldg(reinterpret_cast<const int4 *>(p.bias_i32 + nbase + 4));
                        const float4 s0 = __ldg(reinterpret_cast<const float4 *>(p.m_c + nbase));
                        const float4 s1 = __ldg(reinterpret_cast<const float4 *>(p.m_c + nbase + 4));
                        accv[0] = b0.x; accv[1] = b0.y; accv[2] = b0.z; accv[3] = b0.w;
                        accv[4] = b1.x; accv[5] = b1.y; accv[6] = b1.z; accv[7] = b1.w;
                        mcv[0] = s0.x; mcv[1] = s0.y; mcv[2] = s0.z; mcv[3] = s0.w;
                        mcv[4] = s1.x; mcv[5] = s1.y; mcv[6] = s1.z; mcv[7] = s1.w;
                    } else {
#pragma unroll
                        for (int jj = 0; jj < G; ++jj) {
                            accv[jj] = nbase + jj < p.C_out ? __ldg(p.bias_i32 + nbase + jj) : 0;
                            mcv[jj] = nbase + jj < p.C_out ? __ldg(p.m_c + nbase + jj) : 0.0f;
                        }
                    }
                    for (int ch = 0; ch < p.nchunks; ++ch) {
                        uint32_t v[G];
                        ptx::tmem_ld8(t_row + (uint32_t)(ch * p.chunk_stride + c0), v);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int jj = 0; jj < G; ++jj) accv[jj] += __float2int_rn(__uint_as_float(v[jj]));
                    }
                    if (m >= p.M || nbase >= p.C_out) continue;
                    uint32_t qw[G / 4] = {};
#pragma unroll
                    for (int jj = 0; jj < G; ++jj) {
                        const int qv = requant_i8_fast(accv[jj], mcv[jj], p.inv_s_y, p.zp_y);
                        qw[jj >> 2] |= (uint32_t)(uint8_t)(int8_t)qv << (8 * (jj & 3));
                    }
                    if (p.out_nhwc) {
                        int8_t *yr = static_cast<int8_t *>(p.y) + (size_t)m * p.C_out + nbase;
                        if (nbase + G <= p.C_out && (p.C_out & (G - 1)) == 0) {
                            *reinterpret_cast<uint2 *>(yr) = make_uint2(qw[0], qw[1]);
                        } else {
#pragma unroll
                            for (int jj = 0; jj < G; ++jj)
                                if (nbase + jj < p.C_out) yr[jj] = (int8_t)(qw[jj >> 2] >> (8 * (jj & 3)));
                        }
                    } else {
                        const size_t plane = (size_t)p.OH * p.out_row_stride;
                        const size_t pix = (size_t)oh * p.out_row_stride + ow;
#pragma unroll
                        for (int jj = 0; jj < G; ++jj) {
                            if (nbase + jj >= p.C_out) continue;
                            static_cast<int8_t *>(p.y)[((size_t)img * p.C_out + nbase + jj) * plane + pix] =
                                (int8_t)(qw[jj >> 2] >> (8 * (jj & 3)));
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce_bar(acc));
        }
    }

    __syncthreads();
    if (warp < kMaxProducersI8 && lane == 0 && aborted(abort_flag)) {
        for (int g = last_g; g >= 0 && g > last_g - S; g -= p.nprod)
            ptx::mbar_wait_bounded(raw_bar(g % S), (g / S) & 1, kWaitLimitNs);
    }
    if (warp == kMmaWarpI8 && lane == 0) {
        if (!ptx::mbar_wait_bounded(drain_bar, 0, kWaitLimitNs)) atomicOr(p.status, 1u);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpI8) {
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

}  // namespace

CUresult encode_plain_map(CUtensorMap *tm, CUtensorMapDataType dt, int rank, const void *ptr, const cuuint64_t *dims,
                          const cuuint64_t *strides, const cuuint32_t *box) {
    const DriverFns &fns = driver_fns();
    if (!fns.ok) return CUDA_ERROR_NOT_FOUND;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fns.tiled(tm, dt, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {

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

// X3: K steps per accumulator chunk (CB channels a step), and the chunks
// of the longest part when the nstage = ksteps / kg stages are split.
int x3_kpc(int CB) { return kX3ChunkTerms / CB > 1 ? kX3ChunkTerms / CB : 1; }
int x3_chunks(int ksteps, int kg, int split, int CB) {
    const int nst = ksteps / kg;
    const int unit_ksteps = (nst + split - 1) / split * kg;
    return (unit_ksteps + x3_kpc(CB) - 1) / x3_kpc(CB);
}

int elem_bytes_of(int variant) {
    return variant == CBS_VARIANT_TC_TF32 || variant == CBS_VARIANT_TC_TF32X3 ? 4 : 2;
}

}  // namespace

// Channels per K step for the INT8 variant (int8 bytes per staging row).
// Channels per INT8 K step: the largest of 64, 32, 16 dividing the padded
// channel count and, for two inputs, the first input's channels (a channel
// block never straddles the two tensors).
int i8_channel_block(int c_in_pad, int c_a) {
    for (int cb : {64, 32})
        if (c_in_pad % cb == 0 && c_a % cb == 0) return cb;
    return 16;
}

// Producer warps for a stage count: the largest of 4, 3, 2 that divides it
// (each stage is then always refilled by the same warp).
int tc_producers(int stages) {
    for (int np = kMaxProducers; np >= 2; --np)
        if (stages >= np && stages % np == 0) return np;
    return 1;
}

// GB300 costs the planner works from (SM cycles, measured with single-SM
// probes): a warp issuing TMA copies gets one box through every ~570 cycles
// whatever its size, and all SMs loading at once fill from L2 at ~70 B/cycle
// each.  An issuing thread that waits on a stage barrier gets one MMA out
// every ~95 cycles and loses ~270 cycles per wait; the tensor pipe itself
// takes 48 cycles per M=128, K=16 bf16 MMA up to N=64 and N/2 beyond (TF32:
// twice that).  Each 128-pixel sub-tile has its own issuing thread, so the
// MMA time of a tile is the larger of one issuer's time and the pipe time
// of all its sub-tiles.
constexpr double kClkPerBox = 570.0, kFillBytesPerClk = 70.0, kClkPerStageWait = 270.0;
constexpr double kClkPerMmaIssue = 95.0;

double tc_pipe_clk(int N, bool tf32) {
    const double c = tf32 ? (double)N : 0.5 * N;
    return c > 48.0 ? c : 48.0;
}

// Two MMA-issuing threads on one 128-pixel tile (issuer split): each takes
// the stages of one parity of the CTA's running stage count, into an
// accumulator of its own.  Needs at least two stages per tile (so each
// accumulator gets one) and both accumulators of both TMEM buffers within
// the 512 columns.  The ring depth is made even where it is used.
bool tc_issuer_split_fits(int mmul, int win, int stages_per_tile, int BN) {
    return mmul == 1 && !win && stages_per_tile >= 2 && 4 * next_pow2(BN) <= 512;
}

double tc_tile_mma_clk(double n_mma, double waits, int mmul, int N, bool tf32) {
    const double issue = n_mma * kClkPerMmaIssue + waits * kClkPerStageWait;
    const double pipe = n_mma * mmul * tc_pipe_clk(N, tf32);
    return issue > pipe ? issue : pipe;
}

// Output bytes per element of a TF32/BF16 layer (float or bfloat16).
int tc_out_bytes(bool tf32) { return tf32 ? 4 : 2; }

// NHWC output goes through staged TMA stores when the output rows are
// 16-byte multiples and no store block can spill into another CTA's N tile.
int tc_store_mode(const cbs_layer_desc &d, int BN, int n_tiles, bool tf32) {
    const int eb = tc_out_bytes(tf32);
    const int cbw = 128 / eb;
    if (d.out_layout != CBS_NHWC || (d.c_out * eb) % 16 != 0) return 0;
    return (n_tiles == 1 || BN % cbw == 0) ? 1 : 0;
}

int tc_bias_smem_bytes(const cbs_layer_desc &d) { return d.c_out <= 1024 ? (d.c_out * 4 + 15) / 16 * 16 : 0; }

// Producer warps for a stage count, at most maxp.
int tc_producers_max(int stages, int maxp) {
    for (int np = maxp; np >= 2; --np)
        if (stages >= np && stages % np == 0) return np;
    return 1;
}

// Window geometry of the windowed A path: padded row width, input rows of
// one window box, and the bytes of one window stage.
// - Stride 1 (odd k, pad k/2, 128-byte channel blocks): one box of R_box
//   input rows of Wp = W + 2 pad pixels; tap (r, s) is the window viewed from
//   row r * Wp + s on.
// - Stride 2 (3x3, pad 1, even W, one channel block of 32 or 64 bytes per
//   pixel, one input): tiles are blocks of tile_h output rows x tile_w output
//   columns (ncol blocks across), computed on a grid of Wp = tile_w + 1
//   positions per row (the last one dropped).  Two boxes per tile: plane 0
//   with the even input rows from the block's first output row oh0 on
//   (R_box = tile_h rows) and plane 1 with the odd ones from oh0 - 1
//   (tile_h + 1 rows), both Wp pairs of pixels wide from pair ow0 - 1 on.  A
//   plane row is read as pairs of pixels, PR = 2 RB bytes per operand row;
//   position q = oh' * Wp + ow' then reads, for every tap, one operand row
//   at a fixed offset from q (the taps of output column ow are pixels
//   2 ow - 1, 2 ow and 2 ow + 1: the second half of pair ow - 1 and both
//   halves of pair ow).
struct TcWindow {
    int Wp, R_box, tiles_per_img;
    int tile_w, tile_h, ncol;  // stride 2: output block of a tile, blocks across
    int s2, PR;             // stride-2 pair window; operand row bytes (RB or 2 RB)
    int a_box_bytes;        // bytes the loads of one window stage bring
    int plane1_off;         // byte offset of plane 1 in a stage (stride 2)
    int stage_bytes;        // one window stage, with spare rows, 1024-byte aligned parts
};
bool tc_window_geometry(const cbs_layer_desc &d, int oh, int RB, int cblocks, int tile_m, TcWindow &w) {
    if (d.stride == 1) {
        if (d.k % 2 == 0 || d.pad != d.k / 2 || RB != 128) return false;
        w.s2 = 0;
        w.PR = RB;
        w.Wp = d.w + 2 * d.pad;
        w.R_box = (tile_m - 1) / w.Wp + 2 + 2 * d.pad;
        if (w.Wp > 256 || w.R_box > 256) return false;
        w.a_box_bytes = w.R_box * w.Wp * RB;
        w.plane1_off = 0;
        // The last taps of the last (dropped) columns read up to k-2 rows
        // past the box: the stage keeps 8 spare rows.
        w.stage_bytes = round_up((w.R_box * w.Wp + 8) * RB, 1024);
    } else if (d.stride == 2) {
        if (d.k != 3 || d.pad != 1 || d.w % 2 || d.h < 2 || cblocks != 1 || (RB != 32 && RB != 64) || d.c_in_b > 0)
            return false;
        w.s2 = 1;
        w.PR = 2 * RB;
        const int ow = d.w / 2;
        // Column blocks: the most output pixels per computed position, then
        // the fewest window bytes per image.
        double best_use = -1.0, best_bytes = 0.0;
        int best_ncol = 0;
        for (int ncol = 1; ncol <= 16 && ncol <= ow; ++ncol) {
            const int tw = (ow + ncol - 1) / ncol, wp = tw + 1, th = tile_m / wp;
            if (th < 1 || wp > 256 || th + 1 > 256) continue;
            const int rblocks = (oh + th - 1) / th;
            const double use = (double)ow * oh / ((double)ncol * rblocks * tile_m);
            const double bytes = (double)ncol * rblocks * (2 * th + 1) * wp * w.PR;
            if (use > best_use * 1.01 || (use > best_use * 0.99 && bytes < best_bytes)) {
                best_use = use;
                best_bytes = bytes;
                best_ncol = ncol;
            }
        }
        if (best_ncol == 0) return false;
        w.ncol = best_ncol;
        w.tile_w = (ow + w.ncol - 1) / w.ncol;
        w.Wp = w.tile_w + 1;
        w.tile_h = tile_m / w.Wp;
        w.R_box = w.tile_h;
        w.a_box_bytes = (2 * w.tile_h + 1) * w.Wp * w.PR;
        // Positions past the block (the dropped column, and the tile's rows
        // past tile_h * Wp) read up to tile_m - tile_h * Wp + Wp + 1 pairs
        // past each plane's box: both keep that many spare pairs, and 8 more.
        const int spare = tile_m - w.tile_h * w.Wp + w.Wp + 8;
        w.plane1_off = round_up((w.tile_h * w.Wp + spare) * w.PR, 1024);
        w.stage_bytes = w.plane1_off + round_up(((w.tile_h + 1) * w.Wp + spare) * w.PR, 1024);
        w.tiles_per_img = w.ncol * ((oh + w.tile_h - 1) / w.tile_h);
        return true;
    } else {
        return false;
    }
    w.tile_w = w.tile_h = w.ncol = 0;
    w.tiles_per_img = (oh * w.Wp + tile_m - 1) / tile_m;
    return true;
}

struct TcConfig {
    int BN, mmul, b_res, kg, stages, nprod, st_mode, extra_bytes, win, SB, kpar;
    TcWindow wg;
    int m_tiles, n_tiles, grid;
    int stage_bytes, b_region, b_tile_stride, a_box_bytes;
    double cycles;
};

// Windowed configuration: one window box per tile and channel block (kept
// for all k*k taps), weights resident or in a ring of SB single-tile slots.
bool tc_config_window(const cbs_layer_desc &d, int oh, int RB, int ksteps, bool tf32, TcConfig &c) {
    const int tile_m = kBM * c.mmul;
    const int cblocks = ksteps / (d.k * d.k);
    if (!tc_window_geometry(d, oh, RB, cblocks, tile_m, c.wg)) return false;
    c.kg = 1;
    c.a_box_bytes = c.wg.a_box_bytes;
    c.stage_bytes = c.wg.stage_bytes;
    const int b_bytes = c.BN * RB;
    c.b_tile_stride = (b_bytes + 1023) / 1024 * 1024;
    c.m_tiles = d.n * c.wg.tiles_per_img;
    c.n_tiles = (d.c_out + c.BN - 1) / c.BN;
    c.st_mode = 0;
    c.extra_bytes = tc_bias_smem_bytes(d);
    int cap = 0;
    for (int sb : {4, 2}) {   // streamed weights: slots of one kernel row (k taps) each
        c.SB = c.b_res ? 0 : sb;
        c.b_region = c.b_res ? ksteps * c.b_tile_stride : c.SB * d.k * c.b_tile_stride;
        const int barrier_bytes = 8 * (2 * 16 + 6 + 2 * c.SB) + 16;
        cap = (kSmemBudget - c.b_region - c.extra_bytes - barrier_bytes) / c.stage_bytes;
        if (cap >= 2 || c.b_res) break;
    }
    if (cap > 6) cap = 6;
    if (cap < 2) return false;
    c.stages = cap;
    c.nprod = tc_producers_max(c.stages, c.b_res ? kMaxProducers : kMaxProducers - 1);
    const long long tiles = (long long)c.m_tiles * c.n_tiles;
    if (c.b_res && c.n_tiles > 1) {
        const long long g = tiles < plan_sms(d) ? tiles : (long long)(plan_sms(d) / c.n_tiles) * c.n_tiles;
        if (g <= 0) return false;
        c.grid = (int)g;
    } else {
        c.grid = (int)(tiles < plan_sms(d) ? tiles : plan_sms(d));
    }
    const double tpc = (double)((tiles + c.grid - 1) / c.grid);
    const int kslices = RB / 32;
    const double mma = tpc * (tc_tile_mma_clk((double)ksteps * kslices, (double)cblocks, c.mmul, c.BN, tf32) +
                              (c.b_res ? 0.0 : (double)(ksteps / d.k) * kClkPerStageWait));
    const double boxes = tpc * cblocks * (c.wg.s2 ? 2 : 1) + (c.b_res ? (double)ksteps : tpc * ksteps);
    const double bytes = tpc * cblocks * (double)c.a_box_bytes + (c.b_res ? (double)ksteps : tpc * ksteps) * b_bytes;
    const double t_box = boxes * 140.0, t_fill = bytes / kFillBytesPerClk;
    const double tma = t_box > t_fill ? t_box : t_fill;
    const double vals = c.mmul == 2 ? (double)c.BN : 0.5 * c.BN;
    const double epi = tpc * (250.0 + 45.0 * vals);
    double cyc = mma > tma ? mma : tma;
    if (epi > cyc) cyc = epi;
    cyc += 1500.0 + (double)c.a_box_bytes / kFillBytesPerClk + 250.0 + 45.0 * vals;
    c.cycles = cyc;
    return true;
}

// Shared-memory layout and cost of one configuration (false if it does not fit).
bool tc_config(const cbs_layer_desc &d, long long M, int oh, int RB, int ksteps, bool tf32, int BN, int mmul,
               int b_res, int kg, int win, int kpar, TcConfig &c) {
    c.BN = BN; c.mmul = mmul; c.b_res = b_res; c.kg = kg; c.win = win; c.SB = 0; c.kpar = kpar;
    if (kpar == 2 && !tc_issuer_split_fits(mmul, win, ksteps / kg, BN)) return false;
    if (win) return kpar == 1 && tc_config_window(d, oh, RB, ksteps, tf32, c);
    if (kg * (b_res ? 1 : 2) > 32) return false;   // one issuing lane per box of a stage
    c.a_box_bytes = kBM * mmul * RB;
    const int b_bytes = BN * RB;
    c.b_tile_stride = (b_bytes + 1023) / 1024 * 1024;
    c.b_region = b_res ? ksteps * c.b_tile_stride : 0;
    c.stage_bytes = kg * c.a_box_bytes + (b_res ? 0 : kg * c.b_tile_stride);
    c.m_tiles = (int)((M + kBM * mmul - 1) / (kBM * mmul));
    c.n_tiles = (d.c_out + BN - 1) / BN;
    c.st_mode = tc_store_mode(d, BN, c.n_tiles, tf32);
    c.extra_bytes = (c.st_mode ? kEpiWarps * kStageBlockBytes : 0) + tc_bias_smem_bytes(d);
    const int barrier_bytes = 8 * (2 * 16 + 6) + 16;
    int cap = (kSmemBudget - c.b_region - c.extra_bytes - barrier_bytes) / c.stage_bytes;
    if (cap > 16) cap = 16;
    if (cap < 2) return false;
    c.stages = cap >= 4 ? cap - cap % 4 : cap;
    if (kpar == 2) c.stages -= c.stages & 1;   // even: each ring slot then always feeds the same issuer
    c.nprod = tc_producers(c.stages);
    const long long tiles = (long long)c.m_tiles * c.n_tiles;
    if (b_res && c.n_tiles > 1) {
        // Every CTA keeps one N tile: the grid is a multiple of n_tiles.
        const long long g = tiles < plan_sms(d) ? tiles : (long long)(plan_sms(d) / c.n_tiles) * c.n_tiles;
        if (g <= 0) return false;
        c.grid = (int)g;
    } else {
        c.grid = (int)(tiles < plan_sms(d) ? tiles : plan_sms(d));
    }
    const double tpc = (double)((tiles + c.grid - 1) / c.grid);   // tiles of the busiest CTA
    const int kslices = RB / 32;
    // With the issuer split each issuer takes half the MMAs and waits; the
    // tensor pipe still runs all of them.
    const double mma = tpc * tc_tile_mma_clk((double)ksteps * kslices / kpar, (double)(ksteps / kg) / kpar,
                                             mmul * kpar, BN, tf32);
    const double boxes = tpc * ksteps * (b_res ? 1.0 : 2.0) + (b_res ? (double)ksteps : 0.0);
    const double bytes = tpc * ksteps * (double)(c.a_box_bytes + (b_res ? 0 : b_bytes)) + (b_res ? (double)ksteps * b_bytes : 0.0);
    // Boxes of one stage go out from parallel lanes; the SM's TMA engine
    // still takes ~140 cycles per box.
    const double t_box = boxes * 140.0, t_fill = bytes / kFillBytesPerClk;
    const double tma = t_box > t_fill ? t_box : t_fill;
    // Epilogue: one thread per pixel and 16-column group; eight warps cover
    // two sub-tiles, or split one sub-tile's columns.
    const double vals = mmul == 2 ? (double)BN : 0.5 * BN;
    // (the issuer split reads and adds a second accumulator)
    const double epi = tpc * (250.0 + ((c.st_mode ? 25.0 : 45.0) + (kpar == 2 ? 10.0 : 0.0)) * vals);
    double cyc = mma > tma ? mma : tma;
    if (epi > cyc) cyc = epi;
    // Pipeline fill: the first stage's loads (and a resident weight tile)
    // arrive before any MMA, and the last tile's epilogue follows the last.
    cyc += 1500.0 + (b_res ? kClkPerBox + (double)ksteps * b_bytes / kFillBytesPerClk / c.nprod : 0.0) + 250.0 + 45.0 * vals;
    c.cycles = cyc;
    return true;
}

cbs_status plan_tc(cbs_plan_t &p) {
    const cbs_layer_desc &d = p.desc;
    const bool i8 = p.variant == CBS_VARIANT_TC_INT8;
    const bool x3 = p.variant == CBS_VARIANT_TC_TF32X3;   // FP32 through the staged kernel
    const bool tf32 = p.variant == CBS_VARIANT_TC_TF32;
    const int eb = i8 ? 1 : elem_bytes_of(p.variant);
    int RB, CB, nchunks = 1;
    if (i8) {
        // int8 codes in memory, widened to bf16 operands in shared memory.
        p.c_in_pad = round_up(d.c_in, 16);
        CB = i8_channel_block(p.c_in_pad, d.c_in_b > 0 ? d.c_in - d.c_in_b : p.c_in_pad);
        RB = 2 * CB;
        const int ksteps = d.k * d.k * (p.c_in_pad / CB);
        nchunks = ceil_div(ksteps, 1024 / CB);
    } else {
        // One K step carries RB bytes of channels (32, 64 or 128: a TMA
        // swizzle span); C_in is padded so a pixel holds a multiple of 32 bytes.
        p.c_in_pad = round_up(d.c_in, 32 / eb);
        // Two inputs: a channel block must not straddle them, so RB also
        // divides the first input's pixel bytes (a multiple of 32).
        const int cbytes = p.c_in_pad * eb;
        const int abytes = d.c_in_b > 0 ? (d.c_in - d.c_in_b) * eb : cbytes;
        RB = (cbytes % 128 == 0 && abytes % 128 == 0) ? 128 : (cbytes % 64 == 0 && abytes % 64 == 0) ? 64 : 32;
        CB = RB / eb;
    }
    p.k_gemm = d.k * d.k * p.c_in_pad;
    p.x_bytes = (size_t)d.n * d.h * d.w * p.c_in_pad * eb;
    // X3: weight heads in rows 0..C_out-1, tails in rows C_out..2 C_out-1.
    p.w_packed_bytes = (size_t)d.c_out * p.k_gemm * (x3 ? 8 : (tf32 ? 4 : 2));
    if (d.pad > 127 || (p.oh - 1) * d.stride - d.pad - d.h + 1 < -128 || (p.ow - 1) * d.stride - d.pad - d.w + 1 < -128)
        return fail(CBS_ERR_UNSUPPORTED, "padding outside the im2col corner range");
    if (d.force_split_k > 1 && i8) return fail(CBS_ERR_UNSUPPORTED, "split-K is not built for the INT8 kernel");
    const long long M = (long long)d.n * p.oh * p.ow;
    const int ksteps = d.k * d.k * (p.c_in_pad / CB);
    p.block_k = CB;
    p.split_k = 1;
    p.workspace_bytes = 0;

    if (i8 || x3) {
        p.m_tiles = ceil_div(M, kBM);
        // TMEM holds two accumulator buffers of nchunks * next_pow2(BN)
        // columns (rounded to a power of two): nchunks * next_pow2(BN) <= 256.
        int max_bn = 256;
        while (max_bn >= 16 && nchunks * max_bn > 256) max_bn /= 2;
        // X3 with NCHW input: flat boxes (window = 1) for stride-1 layers
        // whose output grid is the input grid, with W a multiple of 4 (the
        // boxes start 16-byte aligned) and no tile spanning two images.
        const bool flat_fits = x3 && d.in_layout == CBS_NCHW && d.c_in_b == 0 && d.stride == 1 &&
                               d.k == 2 * d.pad + 1 && d.pad <= 3 && d.w % 4 == 0 &&
                               (d.n == 1 || ((long long)p.oh * p.ow) % kBM == 0) &&
                               (long long)d.n * d.c_in < (1LL << 31);
        if (x3 && d.force_window > 0 && !flat_fits)
            return fail(CBS_ERR_UNSUPPORTED,
                        "flat input boxes need 3xTF32 with one NCHW input, stride 1, k = 2 pad + 1 <= 7, W a "
                        "multiple of 4 and batch 1 or whole 128-pixel tiles per image");
        const bool flat = flat_fits && d.force_window > 0;
        p.window = flat ? 1 : 0;
        // One K step: operand A (INT8: bf16; X3: the tail), the weights
        // (X3: head and tail), the staging tile (int8 codes; X3: fp32, the
        // head once converted).  A flat box lands over the A tail and head.
        auto kstep_bytes_of = [&](int c) {
            return kBM * RB + (x3 ? 2 : 1) * round_up(c * RB, 1024) + round_up(kBM * (x3 ? RB : CB), 1024);
        };
        static_assert(kFlatBoxW <= 2 * kBM, "a flat box (kFlatBoxW x CB floats) fits the A tail and head tiles");
        // K steps per stage: the MMA issuer waits twice per stage, so a stage
        // carries the most K steps (up to 4, dividing the K steps) that still
        // leave two stages in shared memory; a split needs at least as many
        // stages per tile as parts.
        auto kgroup_of = [&](int c, int want_split) {
            if (flat) return 1;   // the box lands over the stage's one K step of A tiles
            const int kb = kstep_bytes_of(c);
            for (int g = 4; g >= 1; --g) {
                if (d.force_k_group > 0 && g != d.force_k_group) continue;
                if (want_split > 1 && d.force_k_group <= 0 && g > 1 && ksteps / g < want_split) continue;
                if (ksteps % g == 0 && ((200 * 1024) / (g * kb) >= 2 || g == 1 || d.force_k_group > 0)) return g;
            }
            return 1;
        };
        if (d.force_block_n > 0) {
            const int c = d.force_block_n;
            if (c % 16 || c < 16 || c > 256) return fail(CBS_ERR_INVALID_ARG, "block_n %d: 16..256, multiple of 16", c);
            if (c > max_bn)
                return fail(CBS_ERR_UNSUPPORTED, "block_n %d with %d exact-sum chunks exceeds TMEM", c, nchunks);
        }
        const int full = round_up(d.c_out, 16) < max_bn ? round_up(d.c_out, 16) : max_bn;
        if (full < 16) return fail(CBS_ERR_UNSUPPORTED, "INT8: %d exact-sum chunks exceed TMEM", nchunks);
        // N tile (and X3 split-K parts) from waves of work units over the
        // SMs x the cost of a unit:
        //   INT8: the MMAs of a tile (flat below N = 64);
        //   X3:   per K step, a fixed share for loading and splitting the A
        //         tile (every N tile repeats it) plus the MMAs, and for a
        //         split the partial tiles written and summed.  A split fills
        //         SMs that a single wave of tiles leaves idle; with a wave or
        //         more, only the fewest parts whose accumulator chunks fit
        //         TMEM with that N tile.
        // Measured on GB300 (X3): at batch 16 the C_out = 128 list layers run
        // 10-13% faster with one N tile of 128 than with two of 64, and
        // 128->128 3x3 at 40x40 takes 68 us in 3 parts of N = 128 against
        // 87 us unsplit with N = 64; at batch 1 the chosen splits are the
        // measured best or within a few percent (e.g. 128->256 3x3 s2 at
        // 20x20: N tile 32 in 4 parts, 14.7 us against 19.8 us on the CUDA
        // cores).
        int BN = d.force_block_n > 0 ? d.force_block_n : full;
        int split = d.force_split_k > 1 ? d.force_split_k : 1;
        {
            double best = 1e300;
            for (int c : {full, 256, 192, 128, 96, 64, 32}) {
                if (c > full || c < 16 || (c == 32 && !x3 && c != full)) continue;
                if (d.force_block_n > 0 && c != d.force_block_n) continue;
                const long long tiles = (long long)p.m_tiles * ((d.c_out + c - 1) / c);
                if (!x3) {
                    const double cost = (double)((tiles + plan_sms(d) - 1) / plan_sms(d)) * (c > 64 ? c : 64);
                    if (cost < best * 0.99) { best = cost; BN = c; }
                    continue;
                }
                const bool forced = d.force_split_k >= 1;
                const int sp0 = forced ? d.force_split_k : 1;
                const int sp1 = forced ? d.force_split_k : 16;
                for (int sp = sp0; sp <= sp1; ++sp) {
                    const int g = kgroup_of(c, sp);
                    const int nst = ksteps / g;
                    if (sp > nst) break;
                    // two accumulator buffers of (K-step chunks per part) x N columns in TMEM
                    if (x3_chunks(ksteps, g, sp, CB) * next_pow2(c) > 256) continue;
                    const long long units = tiles * sp;
                    const double cost = (double)((units + plan_sms(d) - 1) / plan_sms(d)) * ((nst + sp - 1) / sp) * g *
                                            (128.0 + c) + (sp > 1 ? 4.0 * sp * c : 0.0);
                    if (cost < best * 0.99) { best = cost; BN = c; split = sp; }
                    // A wave of tiles or more: only the fewest parts whose chunks fit TMEM.
                    if (!forced && tiles >= plan_sms(d)) break;
                }
            }
        }
        p.block_m = kBM;
        p.block_n = BN;
        p.n_tiles = ceil_div(d.c_out, BN);
        p.b_resident = 0;
        const int kstep_bytes = kstep_bytes_of(BN);
        const int kg = kgroup_of(BN, split);
        if (x3 && x3_chunks(ksteps, kg, split, CB) * next_pow2(BN) > 256)
            return fail(CBS_ERR_UNSUPPORTED, "3xTF32: %d K-step chunks of N = %d exceed TMEM (split K or narrow N)",
                        x3_chunks(ksteps, kg, split, CB), BN);
        if (d.force_k_group > 0 && kg != d.force_k_group)
            return fail(CBS_ERR_UNSUPPORTED, "INT8: k_group %d does not divide %d K steps", d.force_k_group, ksteps);
        p.k_group = kg;
        const int stage = kg * kstep_bytes;
        int stages = (200 * 1024) / stage;
        if (stages > 32) stages = 32;
        if (stages < 2) {
            if (2 * stage > kSmemBudget)
                return fail(CBS_ERR_UNSUPPORTED, "two stages of %d K steps do not fit shared memory", kg);
            stages = 2;
        }
        int nprod = kMaxProducersI8;
        while (nprod > 1 && (stages < 2 * nprod)) nprod /= 2;
        stages = stages / nprod * nprod;
        p.stages = stages;
        static_assert(StagedLayout<kStagedX3, kX3Gather>::kThreads == StagedLayout<kStagedX3, kX3Flat>::kThreads,
                      "the NCHW modes launch the same threads");
        p.threads = i8 ? StagedLayout<kStagedI8>::kThreads
                       : d.in_layout == CBS_NCHW ? StagedLayout<kStagedX3, kX3Gather>::kThreads   // 8 converter warps
                                                 : StagedLayout<kStagedX3>::kThreads;
        p.smem_bytes = 1024 + stages * stage + 8 * (3 * stages + 5) + 16;
        const long long tiles = (long long)p.m_tiles * p.n_tiles;
        // X3 split-K: the K stages of a tile in `split` parts, partial tiles
        // in the workspace, summed in order by the last part.
        if (split > ksteps / kg)
            return fail(CBS_ERR_UNSUPPORTED, "split-K %d exceeds the %d pipeline stages of a tile", split, ksteps / kg);
        p.split_k = split;
        if (split > 1)
            p.workspace_bytes = (size_t)round_up((int)tiles * kSplitCounterSlots * 4, 256) +
                                (size_t)tiles * split * kBM * BN * 4;
        const long long units = tiles * split;
        p.grid_ctas = (int)(units < plan_sms(d) ? units : plan_sms(d));
        return CBS_OK;
    }

    // TF32 / BF16: search N tile, sub-tiles per tile, resident weights and
    // K steps per stage with the cost model above.
    int bn_list[12], nbn = 0;
    if (d.force_block_n > 0) {
        const int BN = d.force_block_n;
        if (BN % 16 || BN < 16 || BN > 256) return fail(CBS_ERR_INVALID_ARG, "block_n %d: 16..256, multiple of 16", BN);
        bn_list[nbn++] = BN;
    } else {
        const int full = round_up(d.c_out, 16) < 256 ? round_up(d.c_out, 16) : 256;
        const int cands[] = {full, 256, 192, 128, 96, 64, 48, 32, 16};
        for (int c : cands)
            if (c <= full) {
                bool dup = false;
                for (int k = 0; k < nbn; ++k) dup |= bn_list[k] == c;
                if (!dup) bn_list[nbn++] = c;
            }
    }
    TcConfig best{};
    best.cycles = 1e300;
    for (int bi = 0; bi < nbn; ++bi) {
        const int BN = bn_list[bi];
        for (int mmul = 1; mmul <= 2; ++mmul) {
            if (mmul * next_pow2(BN) > 256) continue;           // two buffers of mmul * BN columns in TMEM
            if (d.force_block_m > 0 && d.force_block_m != kBM * mmul) continue;
            for (int b_res = 0; b_res <= 1; ++b_res) {
                if ((d.force_b_resident > 0 && !b_res) || (d.force_b_resident < 0 && b_res)) continue;
                if (b_res && d.force_split_k > 1 && d.force_b_resident <= 0) continue;   // split-K streams weights
                for (int win = 0; win <= 1; ++win) {
                    // Windowed A moves ~4x fewer bytes from L2 but measured no
                    // faster on GB300 (the MMA rate bounds these layers): it is
                    // used when asked for.
                    if ((d.force_window <= 0 && win) || (d.force_window > 0 && !win)) continue;
                    if (win && d.force_k_group > 0) continue;     // K groups belong to the im2col path
                    for (int kg = 1; kg <= (d.force_k_group > 4 ? d.force_k_group : 4); ++kg) {
                        if (ksteps % kg) continue;
                        // a forced split needs at least that many stages per tile
                        if (d.force_split_k > 1 && d.force_k_group <= 0 && ksteps / kg < d.force_split_k) continue;
                        if (win && kg > 1) break;                  // a window stage is one channel block
                        if (d.force_k_group > 0 && kg != d.force_k_group) continue;
                        for (int kpar = 1; kpar <= 2; ++kpar) {
                            // The issuer split on request only: measured on the
                            // list layers at batch 16 it beat the best one-issuer
                            // plan on 2 of the 19 it applies to (by 3-4%) and lost
                            // up to 64% on the others: 256-pixel tiles share each
                            // weight box between two sub-tiles, the split does not.
                            if ((d.force_issuer_split > 0) != (kpar == 2)) continue;
                            if (kpar == 2 && d.force_split_k > 1) continue;   // split-K keeps one issuer per tile
                            TcConfig c;
                            if (!tc_config(d, M, p.oh, RB, ksteps, tf32, BN, mmul, b_res, kg, win, kpar, c)) continue;
                            if (c.cycles < best.cycles * 0.99) best = c;
                        }
                    }
                }
            }
        }
    }
    if (best.cycles >= 1e299) {
        if (d.force_issuer_split > 0)
            return fail(CBS_ERR_UNSUPPORTED, "no configuration takes the issuer split (block_m 128, im2col A, no "
                                             "split-K, two or more stages per tile, N tile <= 128)");
        return fail(CBS_ERR_UNSUPPORTED, "no tensor-core tile configuration fits shared memory");
    }
    // Split-K on request only.  A launch with fewer tiles than SMs leaves
    // SMs idle, and splitting K over S parts balances the MMAs (e.g. 100
    // tiles of 256x128 over 152 SMs: 288 -> 192 MMAs on the busiest SM at
    // S = 3), but on GB300 the partial tiles cost more than that: the last
    // warp of each region reads every part back at the end of the kernel,
    // and the 128->128 3x3 40x40 BF16 layer at batch 16 went from 24.6 us to
    // 46.2 us.  So the cost model keeps S = 1.
    const int tiles = best.m_tiles * best.n_tiles;
    const int nstage = best.win ? 0 : ksteps / best.kg;
    int split = 1;
    if (d.force_split_k > 1) {
        if (best.win || best.b_res)
            return fail(CBS_ERR_UNSUPPORTED, "split-K needs im2col A and streamed weights (force_window/b_resident)");
        if (d.force_split_k > nstage)
            return fail(CBS_ERR_UNSUPPORTED, "split-K %d exceeds the %d pipeline stages of a tile", d.force_split_k, nstage);
        split = d.force_split_k;
    }
    p.split_k = split;
    if (split > 1) {
        best.grid = tiles * split < plan_sms(d) ? tiles * split : plan_sms(d);
        p.workspace_bytes = (size_t)round_up(tiles * kSplitCounterSlots * 4, 256) +
                            (size_t)tiles * split * (kBM * best.mmul) * best.BN * 4;
    }
    p.block_m = kBM * best.mmul;
    p.block_n = best.BN;
    p.k_group = best.win ? best.SB : best.kg;   // windowed plans: weight-ring slots
    p.b_resident = best.b_res;
    p.window = best.win;
    p.issuer_split = best.kpar;
    p.stages = best.stages;
    p.m_tiles = best.m_tiles;
    p.n_tiles = best.n_tiles;
    p.grid_ctas = best.grid;
    p.threads = kThreads;
    p.smem_bytes = 1024 + best.b_region + best.stages * best.stage_bytes + best.extra_bytes +
                   8 * (2 * best.stages + 6 + 2 * best.SB) + 16;
    return CBS_OK;
}

cbs_status launch_tc(const cbs_plan_t &pl, const void *x, const void *x_b, const void *w_packed, const void *bias,
                     const float *m_c, float inv_s_y, const void *residual, void *y, void *workspace,
                     cudaStream_t s) {
    const cbs_layer_desc &d = pl.desc;
    const DriverFns &fns = driver_fns();
    if (!fns.ok) return fail(CBS_ERR_CUDA, "cannot resolve cuTensorMapEncode* from the driver");
    const bool i8 = pl.variant == CBS_VARIANT_TC_INT8;
    const bool x3 = pl.variant == CBS_VARIANT_TC_TF32X3;
    const bool staged = i8 || x3;                                  // tc_conv_staged_kernel
    const bool f32ops = pl.variant == CBS_VARIANT_TC_TF32 || x3;   // 32-bit operands
    if (pl.variant != CBS_VARIANT_TC_TF32 && pl.variant != CBS_VARIANT_TC_BF16 && !staged)
        return fail(CBS_ERR_UNSUPPORTED, "variant %d", pl.variant);
    const int eb_x = i8 ? 1 : elem_bytes_of(pl.variant);          // activation bytes in memory
    const int eb_w = f32ops ? 4 : 2;                              // operand bytes in shared memory
    const CUtensorMapDataType dt_x = f32ops ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapDataType dt_w = f32ops ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
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
    const int c_a = d.c_in - d.c_in_b;             // channels of the first input (all of them with one)
    if (d.c_in_b > 0) {
        if (!x_b || c_a % CB) return fail(CBS_ERR_PLAN_MISMATCH, "two-input plan: channel blocks");
        P.ca_blocks = c_a / CB;
    } else {
        P.ca_blocks = P.cblocks;
    }
    P.BN = BN; P.stages = pl.stages;
    P.m_tiles = pl.m_tiles; P.n_tiles = pl.n_tiles;
    const int mmul = staged ? 1 : pl.block_m / kBM;
    if (pl.block_m != kBM * mmul || mmul < 1 || mmul > 2) return fail(CBS_ERR_PLAN_MISMATCH, "block_m %d", pl.block_m);
    P.mmul = mmul;
    P.win = staged ? 0 : pl.window;
    P.split = pl.split_k < 1 ? 1 : pl.split_k;
    if (P.split > 1) {
        if (i8 || P.win || pl.b_resident)
            return fail(CBS_ERR_PLAN_MISMATCH, "split-K plan with windowed A, resident weights or INT8");
        if (!workspace) return fail(CBS_ERR_WORKSPACE, "split-K plan without a workspace");
        const size_t counter_bytes = (size_t)round_up(pl.m_tiles * pl.n_tiles * kSplitCounterSlots * 4, 256);
        P.counters = static_cast<unsigned int *>(workspace);
        P.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + counter_bytes);
    }
    P.kg = P.win ? 1 : pl.k_group;
    P.b_res = staged ? 0 : pl.b_resident;
    P.SB = (P.win && !P.b_res) ? pl.k_group : 0;
    if (P.kg < 1 || P.ksteps % P.kg) return fail(CBS_ERR_PLAN_MISMATCH, "k_group %d", pl.k_group);
    if (P.win && !P.b_res && (P.SB < 1 || P.SB > 32)) return fail(CBS_ERR_PLAN_MISMATCH, "weight ring %d", P.SB);
    P.bnp = next_pow2(BN);
    P.kpar = staged ? 1 : pl.issuer_split;
    if (P.kpar != 1 && P.kpar != 2) return fail(CBS_ERR_PLAN_MISMATCH, "issuer_split %d", pl.issuer_split);
    if (P.kpar == 2 && (staged || P.split > 1 || P.stages % 2 || !tc_issuer_split_fits(mmul, P.win, P.ksteps / P.kg, BN)))
        return fail(CBS_ERR_PLAN_MISMATCH, "issuer split with block_m %d, window %d, split-K %d, %d stages, N tile %d",
                    pl.block_m, P.win, P.split, P.stages, BN);
    P.a_bytes = kBM * RB; P.b_bytes = BN * RB;
    P.a_box_bytes = kBM * mmul * RB;
    P.b_tile_stride = round_up(P.b_bytes, 1024);
    P.b_region = P.b_res ? P.ksteps * P.b_tile_stride : P.SB * d.k * P.b_tile_stride;
    if (P.win) {
        TcWindow wg;
        if (!tc_window_geometry(d, pl.oh, RB, P.cblocks, kBM * mmul, wg))
            return fail(CBS_ERR_PLAN_MISMATCH, "window geometry");
        P.Wp = wg.Wp;
        P.R_box = wg.R_box;
        P.tiles_per_img = wg.tiles_per_img;
        P.a_box_bytes = wg.a_box_bytes;
        P.s2 = wg.s2;
        P.PR = wg.PR;
        P.plane1_off = wg.plane1_off;
        P.tile_w = wg.tile_w;
        P.tile_h = wg.tile_h;
        P.ncol = wg.ncol;
        P.swz_a = desc_swizzle_code(wg.PR);
        P.stage_bytes = wg.stage_bytes;
        if (pl.m_tiles != d.n * wg.tiles_per_img) return fail(CBS_ERR_PLAN_MISMATCH, "window tiles");
    }
    if (staged) {
        int nprod = kMaxProducersI8;
        while (nprod > 1 && (pl.stages < 2 * nprod || pl.stages % nprod != 0)) nprod /= 2;
        P.nprod = nprod;
        P.stage_bytes = P.kg * (P.a_bytes + (x3 ? 2 : 1) * P.b_tile_stride + round_up(kBM * XB, 1024));
        if (1024 + pl.stages * P.stage_bytes + 8 * (3 * pl.stages + 5) + 16 > pl.smem_bytes)
            return fail(CBS_ERR_PLAN_MISMATCH, "plan's shared memory does not hold its stages");
    } else {
        P.nprod = P.win ? tc_producers_max(pl.stages, P.b_res ? kMaxProducers : kMaxProducers - 1)
                        : tc_producers(pl.stages);
        if (!P.win) P.stage_bytes = P.kg * P.a_box_bytes + (P.b_res ? 0 : P.kg * P.b_tile_stride);
        const bool tf32 = pl.variant == CBS_VARIANT_TC_TF32;
        P.st_mode = (P.win || P.split > 1) ? 0 : tc_store_mode(d, BN, pl.n_tiles, tf32);
        P.cbw = 128 / tc_out_bytes(tf32);
        P.nblk = (P.BN + P.cbw - 1) / P.cbw;
        P.stg_bytes_total = P.st_mode ? kEpiWarps * kStageBlockBytes : 0;
        P.bias_bytes_smem = tc_bias_smem_bytes(d);
        P.bias_smem = P.bias_bytes_smem > 0;
        P.bias_half = P.bias_smem && d.activation != CBS_ACT_IDENTITY;
        if (1024 + P.b_region + pl.stages * P.stage_bytes + P.stg_bytes_total + P.bias_bytes_smem +
                8 * (2 * pl.stages + 6 + 2 * P.SB) + 16 > pl.smem_bytes)
            return fail(CBS_ERR_PLAN_MISMATCH, "plan's shared memory does not hold its stages");
        if (P.b_res && P.n_tiles > 1 && pl.grid_ctas % P.n_tiles)
            return fail(CBS_ERR_PLAN_MISMATCH, "resident weights need a grid that is a multiple of the N tiles");
    }
    if (i8) {
        P.stg_bytes = kBM * CB;
        P.kpc = 1024 / CB;
        P.nchunks = ceil_div(P.ksteps, P.kpc);
        P.stg_mask = XB == 64 ? 3u : XB == 32 ? 1u : 0u;
        P.op_mask = RB == 128 ? 7u : RB == 64 ? 3u : 1u;
        P.bias_i32 = static_cast<const int32_t *>(bias);
        P.m_c = m_c;
        P.inv_s_y = inv_s_y;
        P.zp_x = d.zero_point_x;
        P.zp_y = d.zero_point_y;
        P.in_h = d.h;
        P.in_w = d.w;
    } else if (x3) {
        if (d.in_layout == CBS_NCHW) {
            // NCHW input: the converter warps read x themselves (no A boxes),
            // or split the flat boxes the producers load.
            if (d.c_in_b > 0) return fail(CBS_ERR_PLAN_MISMATCH, "two-input 3xTF32 plan with NCHW input");
            P.x_nchw = static_cast<const float *>(x);
            P.c_in = d.c_in;
            P.in_h = d.h;
            P.in_w = d.w;
            if (pl.window) {
                if (d.stride != 1 || d.k != 2 * d.pad + 1 || d.pad > 3 || d.w % 4 || pl.oh != d.h || pl.ow != d.w ||
                    (d.n > 1 && P.OHW % kBM) || P.kg != 1)
                    return fail(CBS_ERR_PLAN_MISMATCH, "flat input boxes for this shape");
                P.raw_bytes = kFlatBoxW * CB * 4;   // over the A tail (kBM * RB bytes) and into the head
            }
        } else if (pl.window) {
            return fail(CBS_ERR_PLAN_MISMATCH, "3xTF32 flat input boxes with NHWC input");
        }
        P.stg_bytes = kBM * XB;     // fp32 staging rows, swizzled like the operands (XB = RB)
        P.kpc = x3_kpc(CB);
        P.nchunks = x3_chunks(P.ksteps, P.kg, P.split, CB);
        P.stg_mask = P.op_mask = RB == 128 ? 7u : RB == 64 ? 3u : 1u;
        P.bias = static_cast<const float *>(bias);
    } else {
        P.nchunks = 1;
        P.bias = static_cast<const float *>(bias);
    }
    P.im2col = !(d.k == 1 && d.stride == 1 && d.pad == 0);
    P.out_nhwc = d.out_layout == CBS_NHWC;
    P.out_row_stride = pl.out_row_stride;
    const uint32_t fmt = f32ops ? 2u : 1u;  // TF32 : BF16 operands
    P.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
    P.swz = desc_swizzle_code(RB);
    // Two accumulator buffers (double buffering across tiles); INT8 chunks
    // sit at power-of-two column offsets inside a buffer.
    P.chunk_stride = next_pow2(BN);
    {
        const int cols = staged ? P.nchunks * P.chunk_stride : mmul * P.kpar * P.bnp;
        P.acc_stride = next_pow2(cols) < 16 ? 16 : next_pow2(cols);
    }
    P.tmem_cols = (uint32_t)(2 * P.acc_stride < 32 ? 32 : 2 * P.acc_stride);
    if (P.tmem_cols > 512) return fail(CBS_ERR_UNSUPPORTED, "accumulators need %u TMEM columns", P.tmem_cols);
    P.y = y;
    P.act = d.activation;
    P.residual = residual;
    P.status = device_status_word();
    if (!P.status) return fail(CBS_ERR_CUDA, "cannot resolve the device status word");
    if (pl.grid_ctas <= 0) return CBS_OK;

    alignas(64) CUtensorMap tmA, tmB, tmY;
    std::memset(&tmY, 0, sizeof(tmY));
    CUresult r;
    if (P.st_mode) {
        const int eb_y = eb_w;   // output element: float (TF32) or bfloat16 (BF16)
        const cuuint64_t dims[2] = {(cuuint64_t)d.c_out, (cuuint64_t)P.M};
        const cuuint64_t strides[1] = {(cuuint64_t)d.c_out * eb_y};
        const cuuint32_t box[2] = {(cuuint32_t)P.cbw, 32u};
        const cuuint32_t es[2] = {1, 1};
        r = fns.tiled(&tmY, dt_w, 2, y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (y) failed (%d)", (int)r);
    }
    const cuuint32_t estr1[2] = {1, 1};
    const CUtensorMapSwizzle swz_x = XB == 16 ? CU_TENSOR_MAP_SWIZZLE_NONE : swizzle_for(XB);
    // A map of one input tensor holding `chans` channels per pixel (NHWC).
    auto make_a_map = [&](CUtensorMap *tm, const void *ptr, int chans, const char *what) -> cbs_status {
        CUresult res;
        void *gptr = const_cast<void *>(ptr);
        if (P.win) {
            const cuuint64_t dims[4] = {(cuuint64_t)chans, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
            const cuuint64_t strides[3] = {(cuuint64_t)chans * eb_x, (cuuint64_t)d.w * chans * eb_x,
                                           (cuuint64_t)d.h * d.w * chans * eb_x};
            const cuuint32_t box[4] = {(cuuint32_t)CB, (cuuint32_t)P.Wp, (cuuint32_t)P.R_box, 1u};
            const cuuint32_t es4[4] = {1, 1, 1, 1};
            res = fns.tiled(tm, dt_x, 4, gptr, dims, strides, box, es4, CU_TENSOR_MAP_INTERLEAVE_NONE, swz_x,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (res != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (%s window) failed (%d)", what, (int)res);
        } else if (P.im2col) {
            const cuuint64_t dims[4] = {(cuuint64_t)chans, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
            const cuuint64_t strides[3] = {(cuuint64_t)chans * eb_x, (cuuint64_t)d.w * chans * eb_x,
                                           (cuuint64_t)d.h * d.w * chans * eb_x};
            // Bounding box of the window corners: from -pad to (O-1)*stride - pad.
            const int lower[2] = {-d.pad, -d.pad};
            const int upper[2] = {(pl.ow - 1) * d.stride - d.pad - (d.w - 1), (pl.oh - 1) * d.stride - d.pad - (d.h - 1)};
            const cuuint32_t estr[4] = {1, (cuuint32_t)d.stride, (cuuint32_t)d.stride, 1};
            res = fns.im2col(tm, dt_x, 4, gptr, dims, strides, lower, upper, (cuuint32_t)CB, (cuuint32_t)(kBM * mmul),
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz_x, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (res != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeIm2col (%s) failed (%d)", what, (int)res);
        } else {
            const cuuint64_t dims[2] = {(cuuint64_t)chans, (cuuint64_t)P.M};
            const cuuint64_t strides[1] = {(cuuint64_t)chans * eb_x};
            const cuuint32_t box[2] = {(cuuint32_t)CB, (cuuint32_t)(kBM * mmul)};
            res = fns.tiled(tm, dt_x, 2, gptr, dims, strides, box, estr1, CU_TENSOR_MAP_INTERLEAVE_NONE, swz_x,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (res != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (%s) failed (%d)", what, (int)res);
        }
        return CBS_OK;
    };
    // Stride-2 window plane rp (0: even input rows, 1: odd): rows 2 i + rp of
    // every image, each row as W / 2 pairs of pixels (one pair per box row).
    auto make_plane_map = [&](CUtensorMap *tm, int rp) -> cbs_status {
        const size_t pix = (size_t)pl.c_in_pad * eb_x;
        const char *gptr = static_cast<const char *>(x) + (size_t)rp * d.w * pix;
        const cuuint64_t dims[4] = {(cuuint64_t)(2 * pl.c_in_pad), (cuuint64_t)(d.w / 2),
                                    (cuuint64_t)((d.h + 1 - rp) / 2), (cuuint64_t)d.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(2 * pix), (cuuint64_t)(2 * d.w * pix),
                                       (cuuint64_t)((size_t)d.h * d.w * pix)};
        const cuuint32_t box[4] = {(cuuint32_t)(2 * pl.c_in_pad), (cuuint32_t)P.Wp, (cuuint32_t)(P.R_box + rp), 1u};
        const cuuint32_t es4[4] = {1, 1, 1, 1};
        CUresult res = fns.tiled(tm, dt_x, 4, const_cast<char *>(gptr), dims, strides, box, es4,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(P.PR), CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (res != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (window plane %d) failed (%d)", rp, (int)res);
        return CBS_OK;
    };
    alignas(64) CUtensorMap tmA2;
    if (P.s2) {
        CBS_TRY(make_plane_map(&tmA, 0));
        CBS_TRY(make_plane_map(&tmA2, 1));
    } else if (d.c_in_b > 0) {
        CBS_TRY(make_a_map(&tmA, x, c_a, "A"));
        CBS_TRY(make_a_map(&tmA2, x_b, pl.c_in_pad - c_a, "A of x_b"));
    } else if (P.x_nchw && P.raw_bytes) {
        // Flat boxes: x as rows of H W floats, one per (image, channel).
        const cuuint64_t dims[2] = {(cuuint64_t)d.h * d.w, (cuuint64_t)d.n * d.c_in};
        const cuuint64_t strides[1] = {(cuuint64_t)d.h * d.w * 4};
        const cuuint32_t box[2] = {(cuuint32_t)kFlatBoxW, (cuuint32_t)CB};
        const CUresult res = fns.tiled(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(x), dims, strides,
                                       box, estr1, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (res != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (flat NCHW boxes) failed (%d)", (int)res);
        std::memcpy(&tmA2, &tmA, sizeof(tmA));
    } else if (!P.x_nchw) {
        CBS_TRY(make_a_map(&tmA, x, pl.c_in_pad, "A"));
        std::memcpy(&tmA2, &tmA, sizeof(tmA));
    }
    {
        // X3: the weight tails follow the heads as C_out more rows.
        const cuuint64_t dims[2] = {(cuuint64_t)pl.k_gemm, (cuuint64_t)d.c_out * (x3 ? 2 : 1)};
        const cuuint64_t strides[1] = {(cuuint64_t)pl.k_gemm * eb_w};
        const cuuint32_t box[2] = {(cuuint32_t)CB, (cuuint32_t)BN};
        r = fns.tiled(&tmB, dt_w, 2, const_cast<void *>(w_packed), dims, strides, box, estr1,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(RB), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CBS_ERR_CUDA, "cuTensorMapEncodeTiled (B) failed (%d)", (int)r);
    }
    if (P.x_nchw && !P.raw_bytes) {
        // No A boxes: the A parameters hold a valid map that is never read.
        std::memcpy(&tmA, &tmB, sizeof(tmB));
        std::memcpy(&tmA2, &tmB, sizeof(tmB));
    }

    dim3 grid(pl.grid_ctas, 1, 1);  // persistent: each CTA walks tiles blockIdx.x + i * gridDim.x
    if (pl.smem_bytes > kMaxDynSmem) return fail(CBS_ERR_UNSUPPORTED, "plan needs %d bytes of shared memory", pl.smem_bytes);
    cudaError_t e;
    if (pl.variant == CBS_VARIANT_TC_TF32 || pl.variant == CBS_VARIANT_TC_BF16) {
        using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcParams);
        const int mode = P.kpar == 2 ? kModeIssuerSplit : (P.win && P.s2 ? kModeStride2Window : kModePlain);
        const Kern kerns[2][3] = {{tc_conv_kernel<kTF32, kModePlain>, tc_conv_kernel<kTF32, kModeIssuerSplit>,
                                   tc_conv_kernel<kTF32, kModeStride2Window>},
                                  {tc_conv_kernel<kBF16, kModePlain>, tc_conv_kernel<kBF16, kModeIssuerSplit>,
                                   tc_conv_kernel<kBF16, kModeStride2Window>}};
        const Kern kern = kerns[pl.variant == CBS_VARIANT_TC_BF16 ? 1 : 0][mode];
        e = set_max_dyn_smem(kern, pl.smem_bytes);
        if (e == cudaSuccess) e = launch_kernel(kern, grid, kThreads, pl.smem_bytes, s, tmA, tmA2, tmB, tmY, P);
    } else if (i8) {
        auto kern = tc_conv_staged_kernel<kStagedI8, kX3Nhwc>;
        e = set_max_dyn_smem(kern, pl.smem_bytes);
        if (e == cudaSuccess)
            e = launch_kernel(kern, grid, StagedLayout<kStagedI8>::kThreads, pl.smem_bytes, s, tmA, tmA2, tmB, P);
    } else {
        auto kern = !P.x_nchw    ? tc_conv_staged_kernel<kStagedX3, kX3Nhwc>
                    : P.raw_bytes ? tc_conv_staged_kernel<kStagedX3, kX3Flat>
                                  : tc_conv_staged_kernel<kStagedX3, kX3Gather>;
        const int threads = P.x_nchw ? StagedLayout<kStagedX3, kX3Gather>::kThreads : StagedLayout<kStagedX3>::kThreads;
        if (pl.threads != threads) return fail(CBS_ERR_PLAN_MISMATCH, "threads %d", pl.threads);
        e = set_max_dyn_smem(kern, pl.smem_bytes);
        if (e == cudaSuccess) e = launch_kernel(kern, grid, threads, pl.smem_bytes, s, tmA, tmA2, tmB, P);
    }
    return cuda_check(e, "tensor-core kernel launch");
}

}  // namespace cbs
