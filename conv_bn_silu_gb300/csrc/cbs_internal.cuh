// cbs_internal.cuh -- declarations shared by the library's translation units.
// Nothing here is part of the public ABI (include/cbs.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/cbs.h"

namespace cbs {

// GB300: 152 SMs on two dies.  cbs_plan is host-only and makes no CUDA call:
// it plans for the descriptor's num_sms (this count when 0); launches size
// their grids from the plan.
constexpr int kDefaultNumSMs = 152;
inline int plan_sms(const cbs_layer_desc &d) { return d.num_sms > 0 ? d.num_sms : kDefaultNumSMs; }
// SM count of the current device, for the grids of kernels that have no plan
// (packing and glue); the GB300's count if the query fails.
int current_device_sms();
// Process-unique ID of the calling thread's current CUDA context (0 if none).
// A device reset, or a primary context released and made again, gives a new
// ID: addresses of the library's device globals are cached per ID.
cbs_status current_context_id(unsigned long long *id);
// Device address of the status word that bounded waits report into.
unsigned int *device_status_word();
// One CTA whose bounded wait on a barrier nothing arrives at runs out after
// limit_ns (cbs_selftest_wait_timeout).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);
// Dynamic shared memory ceiling set once on every kernel that opts in above
// 48 KB (the sm_100-family per-block maximum).  Each launch asks for its own
// size below it; a fixed ceiling means a launch recorded in a CUDA graph stays
// valid whatever other launches set afterwards.
constexpr int kMaxDynSmem = 227 * 1024;

// Raises `kern`'s dynamic shared memory ceiling to the per-block maximum less
// its static shared memory, and checks that `bytes` fit under it.
template <typename F>
cudaError_t set_max_dyn_smem(F *kern, int bytes) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    const int cap = kMaxDynSmem - (int)fa.sharedSizeBytes;
    if (bytes > cap) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, cap);
}

// Launch options set by cbs_set_launch_options (CBS_LAUNCH_* bits).
int launch_options();

// Launches `kern` on `s`; with CBS_LAUNCH_PDL set, as a programmatic
// dependent launch (it may be scheduled before the preceding kernel in the
// stream completes; the kernel itself waits for that kernel before it
// touches global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (launch_options() & CBS_LAUNCH_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Records a message for the calling thread and returns `s`.
cbs_status fail(cbs_status s, const char *fmt, ...);
// Maps a CUDA error to CBS_ERR_CUDA (with message) or CBS_OK.
cbs_status cuda_check(cudaError_t e, const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Returns the status of `expr` from the calling function unless it is CBS_OK.
#define CBS_TRY(expr)                      \
    do {                                   \
        cbs_status _s = (expr);            \
        if (_s != CBS_OK) return _s;       \
    } while (0)

// ---------------------------------------------------------------- SIMT FP32
// Tile configurations of the CUDA-core kernel (index = plan->block_k slot).
struct SimtTile { int bm, bn, tm, tn; };
constexpr int kSimtBK = 16;
constexpr SimtTile kSimtTiles[] = {
    {128, 128, 8, 8},  // 0: 256 threads
    {128, 64, 8, 8},   // 1: 128 threads
    {64, 64, 4, 4},    // 2: 256 threads
    {128, 32, 4, 4},   // 3: 256 threads
    {256, 16, 4, 4},   // 4: 256 threads
    {64, 128, 4, 8},   // 5: 256 threads
};
constexpr int kNumSimtTiles = sizeof(kSimtTiles) / sizeof(kSimtTiles[0]);

struct SimtLaunch {
    const float *x;
    const float *x_b;     // nullable: second input, channels C_a..C-1 (channel concatenation)
    int C_a;              // channels held by x (= C without x_b)
    const float *w;       // [K][C_out]
    const float *bias;    // [C_out]
    float *y;
    float *partials;      // split-K partial tiles (workspace)
    unsigned int *counters;  // split-K arrival counters (workspace)
    int N, C, H, W, Cout, OH, OW, KS, stride, pad;
    int M, K, k_chunk, split;
    int out_row_stride;
    int tile;             // index into kSimtTiles
    int in_nhwc, out_nhwc;
    int m_tiles, n_tiles;
    int act;                 // cbs_activation
    const float *residual;   // nullable: added after the activation (same layout as y)
};
cudaError_t launch_simt(const SimtLaunch &L, cudaStream_t s);
// Dynamic shared memory of one CUDA-core CTA (tiles + k table).
int simt_smem_bytes(int tile, int k_chunk, int out_nhwc);

// ---------------------------------------------------------------- stem
struct StemLaunch {
    const void *x, *w, *bias;  // w: [C_out][KS*KS*c_pad] float (kind 0) or bf16 (kinds 1, 2)
    const float *m_c;          // INT8 only
    float inv_s_y;             // INT8 only
    void *y;
    int N, C, c_pad, H, W, Cout, OH, OW, KS, stride, pad;
    int in_nhwc, out_nhwc, out_row_stride;
    int kind;                  // 0 float, 1 bf16, 2 int8
    int tf32;                  // float kind: 1 = the TF32 precision (tensor cores allowed), 0 = FP32
    int act;                   // cbs_activation (float kinds)
    const void *residual;      // nullable, element type and layout of y (float kinds)
    int zp_x, zp_y;            // INT8 zero points of input and output codes
    int grid;                  // tensor-core stems: persistent CTAs (the plan's grid_ctas)
};
cudaError_t launch_stem(const StemLaunch &L, cudaStream_t s);
// TF32, BF16 and INT8 stems (4-channel NHWC input, k <= 3, C_out <= 64;
// kind 3 = TF32, 1 = BF16, 2 = INT8) run on the tensor
// cores (when there are fewer than kStemTcMaxPixels output pixels, for 32-bit
// pixel indices): persistent CTAs of 256 threads, 128 output pixels per tile,
// a ring of kStemTcStages A tiles; the others on the CUDA cores.
bool stem_uses_tensor_cores(int kind, int in_nhwc, int c_pad, int ks, int cout, long long pixels);
constexpr int kStemTcStages = 2, kStemTcCtasPerSm = 5;   // measured: 55.6 us vs 57.3 (4 stages, 3 CTAs) for the 640x640 stem at batch 16
constexpr long long kStemTcMaxPixels = (1ll << 31) - 256;
// TF32: a row of 9 taps x 16 bytes spans two 128-byte panels (A and B), two stages.
constexpr int kStemTf32CtasPerSm = 4;
// Two A stages of 5 x 4 KB, B of 5 x 2 KB, bias, mbarriers, TMEM slot, alignment.
constexpr int kStemTf32SmemBytes = 2 * 20480 + 10240 + 64 * 4 + 16 + 16 + 1024;
// CTAs of the tensor-core stem per SM: kStemTcCtasPerSm, fewer when their
// two accumulators (n_mma columns each, allocated as a power of two >= 32)
// would not fit the SM's 512 TMEM columns together.
inline int stem_tc_ctas_per_sm(int cout, int tf32 = 0) {
    const int n_mma = (cout + 15) / 16 * 16;
    const int cols = 2 * n_mma <= 32 ? 32 : (2 * n_mma <= 64 ? 64 : 128);
    const int want = tf32 ? kStemTf32CtasPerSm : kStemTcCtasPerSm;
    return want < 512 / cols ? want : 512 / cols;
}
// A ring + B (64 rows x 128 B) + bias + two mbarriers + TMEM slot + 1 KB for alignment
constexpr int kStemTcSmemBytes = kStemTcStages * 16384 + 8192 + 64 * 4 + 16 + 16 + 1024;
// The 640x640-class BF16 and TF32 stems (3x3, stride 2, pad 1, even input
// width, 16 output channels, NHWC output, no residual) run a kernel of their
// own that walks whole output rows: TMA brings each input row into shared
// memory once, the CTA rewrites it as the rows of the MMA's A operand, and
// each output row is ceil(OW / 128) M=128 MMAs per kernel row.  Kind 1 is
// BF16, 3 TF32; stem_rows_ctas_per_sm CTAs per SM; kStemRowsAhead output rows
// of input loads in flight per CTA.
constexpr int kStemRowsAhead = 3, kStemRowsESlots = 6;
constexpr int kStemRowsThreads = 288;   // warps 0-7: rewrite and epilogue; warp 8: TMA and MMA issue
constexpr int kStemRowsMaxMtiles = 4;   // OW <= 512: two accumulator buffers of 64 columns
inline int stem_rows_ctas_per_sm(int kind) { return kind == 3 ? 1 : 2; }
// Shared memory of the row kernel for an input width w (0 if it does not
// fit): A-row slots, raw input rows, B, bias, barriers, TMEM slot, alignment.
inline int stem_rows_smem_bytes(int kind, int w) {
    const int px = kind == 3 ? 16 : 8, er = 4 * px;
    const int ow = w / 2, mtiles = (ow + 127) / 128;
    if (mtiles > kStemRowsMaxMtiles) return 0;
    const int bytes = kStemRowsESlots * mtiles * 128 * er + (2 * kStemRowsAhead + 1) * ((w * px + 1023) / 1024 * 1024) +
                      3 * 16 * er + 16 * 4 + 8 * (kStemRowsAhead + 2) + 16 + 1024;
    const int cap = kind == 3 ? 227 * 1024 : (228 * 1024) / 2 - 1024;
    return bytes <= cap ? bytes : 0;
}
inline bool stem_s2_kernel_applies(int kind, int ks, int stride, int pad, int w, int cout, int out_nhwc,
                                   bool residual) {
    return (kind == 1 || kind == 3) && ks == 3 && stride == 2 && pad == 1 && (w & 1) == 0 && cout == 16 && out_nhwc &&
           !residual && stem_rows_smem_bytes(kind, w) > 0;
}
// Encodes a tiled TMA tensor map (no swizzle, no interleave, zero fill
// outside the tensor) through the driver's entry point.
CUresult encode_plain_map(CUtensorMap *tm, CUtensorMapDataType dt, int rank, const void *ptr, const cuuint64_t *dims,
                          const cuuint64_t *strides, const cuuint32_t *box);
constexpr int kStemMaxCin = 4, kStemMaxCout = 64, kStemMaxK = 7;

// ---------------------------------------------------------------- misc kernels
struct FoldLaunch {
    const float *w;           // [C_out][C_in][k][k]
    const float *conv_bias;   // nullable
    const float *gamma, *beta, *mean, *var;
    float eps, s_x;
    int C_out, C_in, KS, c_in_pad;
    int variant;              // cbs_variant
    void *w_packed;
    void *bias;               // float or int32
    float *m_c;               // INT8 only
    int z_x;                  // INT8: input zero point (0 = symmetric)
};
cudaError_t launch_fold(const FoldLaunch &L, cudaStream_t s);

// dtype codes for packing: 0 float, 1 bf16, 2 int8 (quantised with s_x)
cudaError_t launch_pack_input(const float *x_nchw, void *out, int N, int C, int H, int W,
                              int c_pad, int to_nhwc, int dtype, float s_x, int zp, cudaStream_t s);

cudaError_t launch_upsample_concat(const void *a, int ca, const void *b, int cb, void *out,
                                   int n, int h, int w, int nhwc, int elem_bytes,
                                   cudaStream_t s);

cudaError_t launch_dequantize_i8(const int8_t *q, void *out, size_t count, float s, int z, int out_bf16,
                                 cudaStream_t st);
cudaError_t launch_quantize_i8(const void *x, int in_bf16, int8_t *q, size_t count, float s, int z, cudaStream_t st);
cudaError_t launch_sppf_pool(const void *x, void *y, int n, int c, int h, int w, int k, int nhwc, int eb,
                             cudaStream_t s);
cudaError_t launch_maxpool(const void *x, void *y, int n, int c, int h, int w, int k, int stride, int pad, int nhwc,
                           int elem_bytes, cudaStream_t s);

// Device-side status word (bounded waits that expired set it).
unsigned int *device_status_word();  // device address for the current device, or nullptr
cbs_status read_and_reset_status(int *status_out, int reset, cudaStream_t s);

// ---------------------------------------------------------------- tensor-core path
struct TcLaunch;  // defined in k_tc.cu
cbs_status launch_tc(const cbs_plan_t &p, const void *x, const void *x_b, const void *w_packed,
                     const void *bias, const float *m_c, float inv_s_y, const void *residual, void *y,
                     void *workspace, cudaStream_t s);
// Host-side tile selection for the tensor-core variants (fills the tile
// fields of the plan); returns CBS_OK or an error.
cbs_status plan_tc(cbs_plan_t &p);

}  // namespace cbs
