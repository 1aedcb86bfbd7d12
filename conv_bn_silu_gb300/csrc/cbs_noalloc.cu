// cbs_noalloc.cu -- the FP32 CUDA-core fused layer for callers that cannot
// allocate device memory.
//
// Some callers hold only the buffers of the operation itself: a plugin
// interface that hands the layer its input and output pointers and no
// workspace, or a latency-bound serving loop that must not allocate after
// start-up (cudaMalloc may synchronise the whole device, and an allocation
// failure would surface in the middle of a request).  The regular entry point
// asks such a caller for split-K scratch it cannot provide.  This entry point
// takes its scratch from a fixed array in device memory that the library
// itself defines: the module loader places it on every GPU that loads the
// library, where it stays until the process exits.  Nothing is allocated at
// call time.
//
// Rules of use:
//  - The scratch holds at most kNoAllocScratchBytes; a plan whose split-K
//    scratch (plan->workspace_bytes) is larger is rejected with
//    CBS_ERR_WORKSPACE.
//  - The first call on a device looks up the array's device address (with
//    that device current) and caches it; make that first call before any
//    stream capture.  The cache is keyed on the device's current context
//    (its process-unique context ID): after a device reset, or once the
//    primary context has been released and made again, the module is loaded
//    afresh, so the next call looks the address up again.
//  - Every call shares the one array and it keeps the last call's contents.
//    Each call zeroes the split-K arrival counters on its stream before its
//    kernel runs.  Calls whose kernels may overlap on the GPU (different
//    streams without ordering, or concurrent host threads) race on the
//    scratch and give wrong results: order them on one stream.
#include <mutex>

#include "cbs_internal.cuh"

namespace cbs {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device

// The scratch array: split-K counters first, then partial tiles.  Host code
// must not use its name as an address; it reads the device address through
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchEntry {
    unsigned long long ctx_id = 0;   // context the address belongs to (0: none yet)
    void *ptr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

cbs_status scratch_for_current_device(void **out) {
    int dev = -1;
    cbs_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != CBS_OK) return st;
    if (dev < 0 || dev >= kMaxDevices) return fail(CBS_ERR_UNSUPPORTED, "device index %d out of range", dev);
    unsigned long long ctx = 0;
    if ((st = current_context_id(&ctx)) != CBS_OK) return st;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchEntry &e = g_scratch[dev];
    if (!e.ptr || ctx == 0 || e.ctx_id != ctx) {
        void *p = nullptr;
        st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)");
        if (st != CBS_OK) return st;
        // The lookup makes the device's primary context current if none was.
        if ((st = current_context_id(&ctx)) != CBS_OK) return st;
        e.ptr = p;
        e.ctx_id = ctx;
    }
    *out = e.ptr;
    return CBS_OK;
}

}  // namespace
}  // namespace cbs

using namespace cbs;

extern "C" {

cbs_status cbs_conv_bn_silu_f32_noalloc(const cbs_plan_t *p, const float *x, const float *w_packed,
                                        const float *bias, float *y, void *stream) {
    if (!p) return fail(CBS_ERR_INVALID_ARG, "plan is NULL");
    if (p->size != sizeof(cbs_plan_t) || p->abi_version != CBS_ABI_VERSION)
        return fail(CBS_ERR_PLAN_MISMATCH, "plan was not made by cbs_plan of this library");
    if (p->variant != CBS_VARIANT_SIMT_FP32)
        return fail(CBS_ERR_UNSUPPORTED, "the allocation-free entry point runs FP32 CUDA-core plans only");
    if (p->desc.activation != CBS_ACT_SILU || p->desc.residual || p->desc.c_in_b)
        return fail(CBS_ERR_UNSUPPORTED,
                    "the allocation-free entry point runs one-input SiLU plans without a residual");
    if (p->workspace_bytes > kNoAllocScratchBytes)
        return fail(CBS_ERR_WORKSPACE, "plan needs %zu bytes of split-K scratch; the built-in scratch holds %zu",
                    p->workspace_bytes, kNoAllocScratchBytes);
    const cbs_layer_desc &d = p->desc;
    if (d.n == 0) return CBS_OK;
    const void *ptrs[4] = {x, w_packed, bias, y};
    const char *names[4] = {"x", "w_packed", "bias", "y"};
    for (int i = 0; i < 4; ++i) {
        if (!ptrs[i]) return fail(CBS_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(ptrs[i])) return fail(CBS_ERR_MISALIGNED, "%s is not 16-byte aligned", names[i]);
    }
    int tile = -1;
    for (int t = 0; t < kNumSimtTiles; ++t)
        if (kSimtTiles[t].bm == p->block_m && kSimtTiles[t].bn == p->block_n) tile = t;
    if (tile < 0) return fail(CBS_ERR_PLAN_MISMATCH, "unknown CUDA-core tile %dx%d", p->block_m, p->block_n);

    SimtLaunch L{};
    L.x = x; L.w = w_packed; L.bias = bias; L.y = y;
    L.x_b = nullptr; L.C_a = d.c_in;
    L.N = d.n; L.C = d.c_in; L.H = d.h; L.W = d.w; L.Cout = d.c_out; L.OH = p->oh; L.OW = p->ow;
    L.KS = d.k; L.stride = d.stride; L.pad = d.pad;
    L.M = d.n * p->oh * p->ow;
    L.K = d.k * d.k * d.c_in;
    L.split = p->split_k;
    L.k_chunk = (L.K + L.split - 1) / L.split;
    L.k_chunk = (L.k_chunk + kSimtBK - 1) / kSimtBK * kSimtBK;
    L.out_row_stride = p->out_row_stride;
    L.tile = tile;
    L.in_nhwc = d.in_layout == CBS_NHWC;
    L.out_nhwc = d.out_layout == CBS_NHWC;
    L.m_tiles = p->m_tiles;
    L.n_tiles = p->n_tiles;
    cudaStream_t s = (cudaStream_t)stream;
    if (L.split > 1) {
        void *scratch = nullptr;
        cbs_status st = scratch_for_current_device(&scratch);
        if (st != CBS_OK) return st;
        const size_t tiles = (size_t)p->m_tiles * p->n_tiles;
        const size_t counter_bytes = (tiles * sizeof(unsigned) + 255) / 256 * 256;
        L.counters = static_cast<unsigned int *>(scratch);
        L.partials = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + counter_bytes);
        // The counters must start at zero; the array keeps whatever the last
        // call left, so clear them on this call's stream.
        st = cuda_check(cudaMemsetAsync(scratch, 0, counter_bytes, s), "clear split-K counters");
        if (st != CBS_OK) return st;
    }
    return cuda_check(launch_simt(L, s), "SIMT kernel launch (allocation-free entry point)");
}

}  // extern "C"
