// cbs_api.cu -- the C ABI (include/cbs.h): planning, argument checks and
// dispatch to the kernels.  Planning is pure host code with no CUDA call.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "cbs_internal.cuh"

namespace cbs {

namespace {
thread_local char g_msg[512] = "";
}

cbs_status fail(cbs_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

cbs_status cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return CBS_OK;
    return fail(CBS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
std::atomic<int> g_launch_options{CBS_LAUNCH_PDL};
}

int launch_options() { return g_launch_options.load(std::memory_order_relaxed); }

namespace {

int round_up(int v, int m) { return (v + m - 1) / m * m; }
int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

size_t elem_bytes(int prec) {
    switch (prec) {
        case CBS_FP32: case CBS_TF32: return 4;
        case CBS_BF16: return 2;
        default: return 1;
    }
}

// Pick the CUDA-core tile and split-K with a throughput model of the kernel:
// per-thread instructions (FMAs, shared-memory loads, gather and loop
// overhead, epilogue) times warps, issued by 4 schedulers per SM at an
// occupancy-dependent rate, over the number of CTA waves; plus the split-K
// partial-tile traffic (written and read back through L2) and a floor set by
// the layer's own input and output bytes at HBM bandwidth.
struct SimtCost { int tile, split; double cycles; };

SimtCost simt_cost(const cbs_layer_desc &d, int oh, int ow, int t, int split) {
    const SimtTile T = kSimtTiles[t];
    const long long M = (long long)d.n * oh * ow;
    const int K = d.k * d.k * d.c_in;
    const int nt = (T.bm / T.tm) * (T.bn / T.tn);
    const int regs = T.tm * T.tn >= 64 ? 152 : (T.tm * T.tn >= 32 ? 80 : 64);
    const int kc = round_up(ceil_div(K, split), kSimtBK);
    const int splits = ceil_div(K, kc);
    const int smem = simt_smem_bytes(t, kc, d.out_layout == CBS_NHWC) + 1024;
    int res = 65536 / (nt * regs);
    if (res > 2048 / nt) res = 2048 / nt;
    if (res > 228 * 1024 / smem) res = 228 * 1024 / smem;
    if (res < 1) res = 1;
    const long long tiles = (long long)ceil_div(M, T.bm) * ceil_div(d.c_out, T.bn);
    const long long ctas = tiles * splits;
    const double a_pt = (double)T.bm * kSimtBK / nt, b_pt = (double)T.bn * kSimtBK / nt;
    const double per_thread = (double)T.tm * T.tn * kc + (double)kc * (T.tm + T.tn) / 4.0 +
                              (double)kc / kSimtBK * (a_pt * 7 + b_pt * 6 + 12) + T.tm * T.tn * 9.0 + 150.0 +
                              (splits > 1 ? T.tm * T.tn * (0.5 * splits + 2) : 0.0);
    const double cta_warp_instr = per_thread * nt / 32.0;
    const long long sms = plan_sms(d);
    const long long slots = sms * res;
    const long long waves = (ctas + slots - 1) / slots;
    const long long per_sm = (ctas + sms - 1) / sms < res ? (ctas + sms - 1) / sms : res;
    const double warps = (double)per_sm * nt / 32.0;
    const double ipc = 4.0 * 0.7 * (warps >= 24 ? 1.0 : warps / 24.0);
    double cycles = (double)waves * per_sm * cta_warp_instr / ipc;
    if (splits > 1) cycles += (double)ctas * T.bm * T.bn * 8.0 / 2600.0;  // partials through L2
    const double io_bytes = 4.0 * ((double)d.n * d.c_in * d.h * d.w + (double)M * d.c_out);
    const double mem_cycles = io_bytes / 3100.0;  // ~6 TB/s at ~1.9 GHz
    if (cycles < mem_cycles) cycles = mem_cycles;
    cycles += 1500.0;  // launch and fill
    return {t, splits, cycles};
}

void plan_simt(cbs_plan_t &p) {
    const cbs_layer_desc &d = p.desc;
    const long long M = (long long)d.n * p.oh * p.ow;
    const int K = d.k * d.k * d.c_in;
    SimtCost best{1, 1, 1e300};
    for (int t = 0; t < kNumSimtTiles; ++t) {
        if (d.force_block_n > 0 && kSimtTiles[t].bn != d.force_block_n) continue;
        if (d.force_block_m > 0 && kSimtTiles[t].bm != d.force_block_m) continue;
        int max_split = K / (kSimtBK * 2) > 1 ? K / (kSimtBK * 2) : 1;
        if (max_split > 32) max_split = 32;
        int lo = 1;
        if (d.force_split_k > 0) lo = max_split = d.force_split_k;
        for (int split = lo; split <= max_split; ++split) {
            const SimtCost c = simt_cost(d, p.oh, p.ow, t, split);
            if (c.cycles < best.cycles) best = c;
        }
    }
    const SimtTile T = kSimtTiles[best.tile];
    p.block_m = T.bm;
    p.block_n = T.bn;
    p.block_k = kSimtBK;
    p.stages = 2;
    p.threads = (T.bm / T.tm) * (T.bn / T.tn);
    p.m_tiles = ceil_div(M, T.bm);
    p.n_tiles = ceil_div(d.c_out, T.bn);
    // K per split, a multiple of BK; recompute the split so none is empty.
    const int kc = round_up(ceil_div(K, d.force_split_k > 0 ? d.force_split_k : best.split), kSimtBK);
    p.split_k = ceil_div(K, kc);
    p.smem_bytes = simt_smem_bytes(best.tile, kc, d.out_layout == CBS_NHWC);
    p.grid_ctas = p.m_tiles * p.n_tiles * p.split_k;
    p.variant = CBS_VARIANT_SIMT_FP32;
    p.workspace_bytes = 0;
    if (p.split_k > 1) {
        const size_t tiles = (size_t)p.m_tiles * p.n_tiles;
        const size_t counters = (tiles * sizeof(unsigned) + 255) / 256 * 256;
        p.workspace_bytes = counters + tiles * p.split_k * (size_t)T.bm * T.bn * sizeof(float);
    }
}

int simt_tile_index(const cbs_plan_t &p) {
    for (int t = 0; t < kNumSimtTiles; ++t)
        if (kSimtTiles[t].bm == p.block_m && kSimtTiles[t].bn == p.block_n) return t;
    return -1;
}

cbs_status check_plan(const cbs_plan_t *p) {
    if (!p) return fail(CBS_ERR_INVALID_ARG, "plan is NULL");
    if (p->size != sizeof(cbs_plan_t) || p->abi_version != CBS_ABI_VERSION)
        return fail(CBS_ERR_PLAN_MISMATCH, "plan was not made by cbs_plan of this library (size %u, abi %u)",
                    p->size, p->abi_version);
    return CBS_OK;
}

cbs_status check_ptr(const void *ptr, const char *name, bool nullable = false) {
    if (!ptr) return nullable ? CBS_OK : fail(CBS_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(ptr)) return fail(CBS_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    return CBS_OK;
}


StemLaunch stem_launch(const cbs_plan_t &p, const void *x, const void *w, const void *bias, const float *m_c,
                       float inv_s_y, void *y) {
    const cbs_layer_desc &d = p.desc;
    StemLaunch L{};
    L.x = x; L.w = w; L.bias = bias; L.m_c = m_c; L.inv_s_y = inv_s_y; L.y = y;
    L.N = d.n; L.C = d.c_in; L.c_pad = p.c_in_pad; L.H = d.h; L.W = d.w; L.Cout = d.c_out;
    L.OH = p.oh; L.OW = p.ow; L.KS = d.k; L.stride = d.stride; L.pad = d.pad;
    L.in_nhwc = d.in_layout == CBS_NHWC;
    L.out_nhwc = d.out_layout == CBS_NHWC;
    L.out_row_stride = p.out_row_stride;
    L.kind = d.prec == CBS_INT8 ? 2 : (d.prec == CBS_BF16 ? 1 : 0);
    L.tf32 = d.prec == CBS_TF32;
    L.act = d.activation;
    L.residual = nullptr;
    L.zp_x = d.prec == CBS_INT8 ? d.zero_point_x : 0;
    L.zp_y = d.prec == CBS_INT8 ? d.zero_point_y : 0;
    L.grid = p.grid_ctas;
    return L;
}

}  // namespace
}  // namespace cbs

using namespace cbs;

extern "C" {

int cbs_abi_version(void) { return CBS_ABI_VERSION; }

cbs_status cbs_set_launch_options(int flags) {
    if (flags & ~CBS_LAUNCH_PDL) return fail(CBS_ERR_INVALID_ARG, "unknown launch option bits 0x%x", flags);
    g_launch_options.store(flags);
    return CBS_OK;
}

int cbs_launch_options(void) { return g_launch_options.load(); }

const char *cbs_last_error(void) { return g_msg; }

const char *cbs_status_string(cbs_status s) {
    switch (s) {
        case CBS_OK: return "CBS_OK";
        case CBS_ERR_INVALID_ARG: return "CBS_ERR_INVALID_ARG";
        case CBS_ERR_UNSUPPORTED: return "CBS_ERR_UNSUPPORTED";
        case CBS_ERR_MISALIGNED: return "CBS_ERR_MISALIGNED";
        case CBS_ERR_WORKSPACE: return "CBS_ERR_WORKSPACE";
        case CBS_ERR_CUDA: return "CBS_ERR_CUDA";
        case CBS_ERR_TIMEOUT: return "CBS_ERR_TIMEOUT";
        case CBS_ERR_PLAN_MISMATCH: return "CBS_ERR_PLAN_MISMATCH";
    }
    return "CBS_ERR_UNKNOWN";
}

cbs_status cbs_plan(const cbs_layer_desc *d, cbs_plan_t *out) {
    if (!d || !out) return fail(CBS_ERR_INVALID_ARG, "desc or plan pointer is NULL");
    const cbs_layer_desc D = *d;
    if (D.n < 0 || D.c_in < 1 || D.c_out < 1 || D.h < 1 || D.w < 1 || D.k < 1 || D.stride < 1 ||
        D.pad < 0)
        return fail(CBS_ERR_INVALID_ARG, "bad shape n=%d c_in=%d c_out=%d h=%d w=%d k=%d stride=%d pad=%d",
                    D.n, D.c_in, D.c_out, D.h, D.w, D.k, D.stride, D.pad);
    if (D.k > 15 || D.stride > 8 || D.pad >= D.k)
        return fail(CBS_ERR_UNSUPPORTED, "k=%d stride=%d pad=%d outside the supported range (k<=15, stride<=8, pad<k)",
                    D.k, D.stride, D.pad);
    if (D.h + 2 * D.pad < D.k || D.w + 2 * D.pad < D.k)
        return fail(CBS_ERR_INVALID_ARG, "filter larger than the padded image");
    if ((D.in_layout != CBS_NCHW && D.in_layout != CBS_NHWC) ||
        (D.out_layout != CBS_NCHW && D.out_layout != CBS_NHWC))
        return fail(CBS_ERR_INVALID_ARG, "unknown layout");
    if (D.prec < CBS_FP32 || D.prec > CBS_INT8) return fail(CBS_ERR_INVALID_ARG, "unknown precision %d", D.prec);
    if (D.activation != CBS_ACT_SILU && D.activation != CBS_ACT_IDENTITY)
        return fail(CBS_ERR_INVALID_ARG, "unknown activation %d", D.activation);
    if (D.residual != 0 && D.residual != 1) return fail(CBS_ERR_INVALID_ARG, "residual must be 0 or 1");
    if (D.prec == CBS_INT8 && (D.activation != CBS_ACT_SILU || D.residual))
        return fail(CBS_ERR_UNSUPPORTED, "INT8: the specified requantising SiLU epilogue only");
    if (D.c_in_b < 0 || D.c_in_b >= D.c_in)
        return fail(CBS_ERR_INVALID_ARG, "c_in_b %d: 0 (one input) or 1..c_in-1 (c_in = %d)", D.c_in_b, D.c_in);
    if (D.prec != CBS_INT8 && (D.zero_point_x || D.zero_point_y))
        return fail(CBS_ERR_INVALID_ARG, "zero points apply to INT8 plans only");
    if (D.num_sms < 0 || D.num_sms > 4096)
        return fail(CBS_ERR_INVALID_ARG, "num_sms %d: 0 (the GB300's 152) or the device's SM count", D.num_sms);
    if (D.zero_point_x < -128 || D.zero_point_x > 127 || D.zero_point_y < -128 || D.zero_point_y > 127)
        return fail(CBS_ERR_INVALID_ARG, "zero points must lie in [-128, 127] (z_x %d, z_y %d)", D.zero_point_x,
                    D.zero_point_y);

    cbs_plan_t p;
    std::memset(&p, 0, sizeof(p));
    p.size = sizeof(cbs_plan_t);
    p.abi_version = CBS_ABI_VERSION;
    p.desc = D;
    p.k_group = 1;
    p.issuer_split = 1;
    p.oh = (D.h + 2 * D.pad - D.k) / D.stride + 1;
    p.ow = (D.w + 2 * D.pad - D.k) / D.stride + 1;
    const long long M = (long long)D.n * p.oh * p.ow;
    if (M > 0x7fffffffLL || (long long)D.n * D.c_in * D.h * D.w > (1LL << 40))
        return fail(CBS_ERR_UNSUPPORTED, "problem too large for 32-bit pixel indexing");

    const bool stem_fits = D.c_in <= kStemMaxCin && D.c_out <= kStemMaxCout && D.k <= kStemMaxK && D.c_in_b == 0;
    int variant = D.force_variant;
    bool auto_x3 = false;
    if (variant < 0) {
        variant = stem_fits ? (int)CBS_VARIANT_STEM : D.prec;  // FP32->SIMT, TF32, BF16, INT8
        // FP32 with NHWC input runs on the tensor cores (3xTF32, within the
        // FP32 bar; split-K where the tiles leave SMs idle).  Measured on
        // GB300 over the list layers: 1.3-3.4x faster than the CUDA cores at
        // batch 16, and faster on every layer at batch 1 (by 2-40%).  Only
        // when every input's channel count is a multiple of 8: the NHWC input
        // then needs no padding and is the same bytes for either kernel.  A
        // descriptor that forces a tile field is tuning the CUDA-core kernel.
        const int c_a = D.c_in - D.c_in_b;
        const bool forces_tiles = D.force_split_k > 0 || D.force_block_n > 0 || D.force_block_m > 0 ||
                                  D.force_k_group > 0 || D.force_b_resident != 0 || D.force_window > 0 ||
                                  D.force_issuer_split > 0;
        if (variant == CBS_VARIANT_SIMT_FP32 && D.in_layout == CBS_NHWC && c_a % 8 == 0 && D.c_in_b % 8 == 0 &&
            !forces_tiles) {
            variant = CBS_VARIANT_TC_TF32X3;
            auto_x3 = true;
        }
        // FP32 with NCHW input: the same kernel, its converter warps reading
        // the NCHW input themselves, when C_in >= 32 and either k >= 3 or
        // C_in >= 64.  Measured per layer at batch 1 against the CUDA cores'
        // best plans, it wins on every list layer but the 16-channel 3x3 (by
        // 10%) and the 32-channel 1x1 (by 5%).
        if (variant == CBS_VARIANT_SIMT_FP32 && D.in_layout == CBS_NCHW && D.c_in_b == 0 && D.c_in % 8 == 0 &&
            D.c_in >= 32 && (D.k >= 3 || D.c_in >= 64) && !forces_tiles) {
            variant = CBS_VARIANT_TC_TF32X3;
            auto_x3 = true;
        }
    }
    if (variant == CBS_VARIANT_STEM) {
        if (!stem_fits)
            return fail(CBS_ERR_UNSUPPORTED, "stem variant needs one input with C_in <= %d, C_out <= %d, k <= %d",
                        kStemMaxCin, kStemMaxCout, kStemMaxK);
    } else {
        const int need_prec[] = {CBS_FP32, CBS_TF32, CBS_BF16, CBS_INT8, -1, CBS_FP32};
        if (variant < 0 || variant > 5 || need_prec[variant] != D.prec)
            return fail(CBS_ERR_INVALID_ARG, "variant %d does not compute precision %d", variant, D.prec);
    }
    p.variant = variant;
    if (D.force_issuer_split < -1 || D.force_issuer_split > 1)
        return fail(CBS_ERR_INVALID_ARG, "force_issuer_split %d: -1, 0 or 1", D.force_issuer_split);
    if (D.force_issuer_split > 0 && variant != CBS_VARIANT_TC_TF32 && variant != CBS_VARIANT_TC_BF16)
        return fail(CBS_ERR_UNSUPPORTED, "the issuer split belongs to the TF32/BF16 tensor-core variants");

    if (D.out_row_stride != 0) {
        if (D.out_layout != CBS_NCHW)
            return fail(CBS_ERR_INVALID_ARG, "out_row_stride applies to NCHW output only");
        if (D.out_row_stride < p.ow)
            return fail(CBS_ERR_INVALID_ARG, "out_row_stride %d < OW %d", D.out_row_stride, p.ow);
    }
    p.out_row_stride = D.out_row_stride ? D.out_row_stride : p.ow;

    const size_t eb = elem_bytes(D.prec);
    if (variant == CBS_VARIANT_STEM) {
        p.c_in_pad = (D.in_layout == CBS_NHWC && D.prec != CBS_FP32) ? 4 : D.c_in;
    } else if (variant == CBS_VARIANT_SIMT_FP32) {
        p.c_in_pad = D.c_in;
    } else {
        // 3xTF32 takes NCHW input too (one input: its converters read it).
        if (D.in_layout != CBS_NHWC && !(variant == CBS_VARIANT_TC_TF32X3 && D.c_in_b == 0))
            return fail(CBS_ERR_UNSUPPORTED, "tensor-core variants read NHWC input (use cbs_pack_input)");
        p.c_in_pad = round_up(D.c_in, (int)(16 / eb));
        // First input: whole channel blocks (32 bytes, INT8: 16 channels); second: TMA strides.
        const size_t a_unit = D.prec == CBS_INT8 ? 16 : 32;
        if (D.c_in_b > 0 && (((size_t)(D.c_in - D.c_in_b) * eb) % a_unit || ((size_t)D.c_in_b * eb) % 16))
            return fail(CBS_ERR_UNSUPPORTED,
                        "two-input tensor-core layers need the first input's pixels to be a multiple of %zu bytes "
                        "and the second's of 16 bytes (c_in %d, c_in_b %d)", a_unit, D.c_in, D.c_in_b);
    }
    p.k_gemm = D.k * D.k * p.c_in_pad;
    p.x_bytes = (size_t)D.n * D.h * D.w * p.c_in_pad * eb;
    if (D.out_layout == CBS_NCHW)
        p.y_bytes = (size_t)D.n * D.c_out * p.oh * p.out_row_stride * eb;
    else
        p.y_bytes = (size_t)M * D.c_out * eb;
    p.w_packed_bytes = (size_t)D.c_out * p.k_gemm * (D.prec == CBS_FP32 || D.prec == CBS_TF32 ? 4 : 2);
    p.bias_bytes = (size_t)D.c_out * 4;

    if (variant == CBS_VARIANT_STEM) {
        const int cout_t = D.c_out <= 16 ? 16 : (D.c_out <= 32 ? 32 : 64);
        // pixels per thread, as the direct kernel picks them (k_stem.cu)
        const int px_per_thread = (D.prec == CBS_FP32 || D.prec == CBS_TF32) ? 1
                                  : D.prec == CBS_INT8 ? (cout_t == 16 ? 4 : (cout_t == 32 ? 2 : 1))
                                                       : (cout_t <= 32 ? 2 : 1);
        p.block_m = 256 * px_per_thread;  // output pixels per CTA: 256 threads, px_per_thread each
        const int tc_kind = D.prec == CBS_BF16 ? 1 : (D.prec == CBS_INT8 ? 2 : (D.prec == CBS_TF32 ? 3 : 0));
        const bool tc = stem_uses_tensor_cores(tc_kind, D.in_layout == CBS_NHWC, p.c_in_pad, D.k, D.c_out, M);
        if (tc) p.block_m = 128;           // tensor-core stem: 128 pixels (one M=128 MMA) per CTA
        p.block_n = cout_t;
        p.block_k = D.k * D.k * p.c_in_pad;
        p.stages = 1;
        p.split_k = 1;
        p.m_tiles = (int)((M + p.block_m - 1) / p.block_m);
        p.n_tiles = 1;
        // the tensor-core stem is persistent: kStemTcCtasPerSm CTAs per SM walk the tiles
        p.grid_ctas = tc ? std::min(p.m_tiles, plan_sms(D) * stem_tc_ctas_per_sm(D.c_out, tc_kind == 3)) : p.m_tiles;
        p.threads = 256;
        p.smem_bytes = tc ? (tc_kind == 3 ? kStemTf32SmemBytes : kStemTcSmemBytes) : D.k * D.k * p.c_in_pad * cout_t * 4;
        if (tc && stem_s2_kernel_applies(tc_kind, D.k, D.stride, D.pad, D.w, D.c_out, D.out_layout == CBS_NHWC,
                                         D.residual != 0)) {
            // the stem's own kernel: one band of output rows per CTA
            p.grid_ctas = std::min(D.n * p.oh, plan_sms(D) * stem_rows_ctas_per_sm(tc_kind));
            p.smem_bytes = stem_rows_smem_bytes(tc_kind, D.w);
            p.threads = kStemRowsThreads;
        }
        p.workspace_bytes = 0;
    } else if (variant == CBS_VARIANT_SIMT_FP32) {
        plan_simt(p);
    } else {
        const cbs_status st = plan_tc(p);
        if (st != CBS_OK) {
            if (!auto_x3) return st;
            // No 3xTF32 configuration for this shape: the CUDA-core kernel.
            cbs_layer_desc simt = D;
            simt.force_variant = CBS_VARIANT_SIMT_FP32;
            CBS_TRY(cbs_plan(&simt, out));
            out->desc.force_variant = D.force_variant;
            return CBS_OK;
        }
        if (p.variant == CBS_VARIANT_TC_TF32X3 && D.in_layout == CBS_NCHW)
            p.x_bytes = (size_t)D.n * D.c_in * D.h * D.w * eb;   // read as given
    }
    if (D.c_in_b > 0) {   // x holds the first c_in - c_in_b channels, x_b the rest (plus padding)
        const int c_a = D.c_in - D.c_in_b;
        const size_t pixels = (size_t)D.n * D.h * D.w;
        p.x_bytes = pixels * c_a * eb;
        p.x_b_bytes = pixels * (size_t)(p.c_in_pad - c_a) * eb;
    }
    *out = p;
    return CBS_OK;
}

cbs_status cbs_fold_bn(const cbs_plan_t *p, const float *w_oihw, const float *conv_bias,
                       const float *gamma, const float *beta, const float *mean, const float *var,
                       float eps, float s_x, void *w_packed, void *bias, float *m_c, void *stream) {
    CBS_TRY(check_plan(p));
    CBS_TRY(check_ptr(w_oihw, "w"));
    CBS_TRY(check_ptr(conv_bias, "conv_bias", true));
    CBS_TRY(check_ptr(gamma, "gamma"));
    CBS_TRY(check_ptr(beta, "beta"));
    CBS_TRY(check_ptr(mean, "mean"));
    CBS_TRY(check_ptr(var, "var"));
    CBS_TRY(check_ptr(w_packed, "w_packed"));
    CBS_TRY(check_ptr(bias, "bias"));
    if (!(eps > 0.0f)) return fail(CBS_ERR_INVALID_ARG, "eps must be > 0");
    if (p->desc.prec == CBS_INT8) {
        CBS_TRY(check_ptr(m_c, "m_c"));
        if (!(s_x > 0.0f)) return fail(CBS_ERR_INVALID_ARG, "s_x must be > 0 for INT8");
    }
    FoldLaunch L;
    L.w = w_oihw; L.conv_bias = conv_bias; L.gamma = gamma; L.beta = beta; L.mean = mean; L.var = var;
    L.eps = eps; L.s_x = s_x;
    L.C_out = p->desc.c_out; L.C_in = p->desc.c_in; L.KS = p->desc.k; L.c_in_pad = p->c_in_pad;
    L.variant = p->variant;
    if (p->variant == CBS_VARIANT_STEM) {  // stem weights use the tensor-core layouts of its precision
        const int by_prec[] = {CBS_VARIANT_TC_TF32, CBS_VARIANT_TC_TF32, CBS_VARIANT_TC_BF16, CBS_VARIANT_TC_INT8};
        L.variant = by_prec[p->desc.prec];
    }
    L.w_packed = w_packed; L.bias = bias; L.m_c = m_c;
    L.z_x = p->desc.prec == CBS_INT8 ? p->desc.zero_point_x : 0;
    return cuda_check(launch_fold(L, (cudaStream_t)stream), "fold kernel launch");
}

cbs_status cbs_pack_input(const cbs_plan_t *p, const float *x_nchw, void *x_packed, float s_x,
                          void *stream) {
    CBS_TRY(check_plan(p));
    CBS_TRY(check_ptr(x_nchw, "x_nchw"));
    CBS_TRY(check_ptr(x_packed, "x_packed"));
    const cbs_layer_desc &d = p->desc;
    if (d.c_in_b > 0)
        return fail(CBS_ERR_UNSUPPORTED, "two-input plan: pack each input with a one-input plan of its own channels");
    if (d.n == 0) return CBS_OK;
    int dtype = 0;
    if (d.prec == CBS_BF16) dtype = 1;
    if (d.prec == CBS_INT8) {
        dtype = 2;
        if (!(s_x > 0.0f)) return fail(CBS_ERR_INVALID_ARG, "s_x must be > 0 for INT8");
    }
    const int to_nhwc = d.in_layout == CBS_NHWC;
    return cuda_check(launch_pack_input(x_nchw, x_packed, d.n, d.c_in, d.h, d.w, p->c_in_pad, to_nhwc,
                                        dtype, s_x, d.prec == CBS_INT8 ? d.zero_point_x : 0, (cudaStream_t)stream),
                      "pack kernel launch");
}

static cbs_status check_conv_common(const cbs_plan_t *p, const void *x, const void *w, const void *bias,
                                    const void *y, const void *ws, size_t ws_bytes) {
    CBS_TRY(check_ptr(x, "x"));
    CBS_TRY(check_ptr(w, "w_packed"));
    CBS_TRY(check_ptr(bias, "bias"));
    CBS_TRY(check_ptr(y, "y"));
    if (p->workspace_bytes > 0) {
        if (!ws) return fail(CBS_ERR_WORKSPACE, "plan needs %zu bytes of workspace, got NULL", p->workspace_bytes);
        if (ws_bytes < p->workspace_bytes)
            return fail(CBS_ERR_WORKSPACE, "workspace %zu bytes < %zu required", ws_bytes, p->workspace_bytes);
        CBS_TRY(check_ptr(ws, "workspace"));
    }
    return CBS_OK;
}

}  // extern "C"

namespace {

// The FP32 / TF32 / BF16 layer with the plan's activation and an optional
// residual (already checked against the plan by the caller).
cbs_status conv_act_impl(const cbs_plan_t *p, const void *x, const void *x_b, const void *w_packed,
                         const float *bias, const void *residual, void *y, void *workspace, size_t workspace_bytes,
                         void *stream) {
    const cbs_layer_desc &d = p->desc;
    if (d.n == 0) return CBS_OK;  // empty batch: nothing is read or written
    CBS_TRY(check_conv_common(p, x, w_packed, bias, y, workspace, workspace_bytes));
    if (d.c_in_b > 0) CBS_TRY(check_ptr(x_b, "x_b"));
    if (residual && !aligned16(residual)) return fail(CBS_ERR_MISALIGNED, "residual is not 16-byte aligned");
    if (p->variant == CBS_VARIANT_STEM) {
        StemLaunch L = stem_launch(*p, x, w_packed, bias, nullptr, 0.0f, y);
        L.residual = residual;
        return cuda_check(launch_stem(L, (cudaStream_t)stream), "stem kernel launch");
    }
    if (p->variant == CBS_VARIANT_SIMT_FP32) {
        SimtLaunch L;
        std::memset(&L, 0, sizeof(L));
        L.x = (const float *)x; L.w = (const float *)w_packed; L.bias = bias; L.y = (float *)y;
        L.x_b = d.c_in_b > 0 ? (const float *)x_b : nullptr;
        L.C_a = d.c_in - d.c_in_b;
        L.N = d.n; L.C = d.c_in; L.H = d.h; L.W = d.w; L.Cout = d.c_out; L.OH = p->oh; L.OW = p->ow;
        L.KS = d.k; L.stride = d.stride; L.pad = d.pad;
        L.M = d.n * p->oh * p->ow;
        L.K = d.k * d.k * d.c_in;
        L.split = p->split_k;
        L.k_chunk = (L.K + L.split - 1) / L.split;
        L.k_chunk = (L.k_chunk + kSimtBK - 1) / kSimtBK * kSimtBK;
        L.out_row_stride = p->out_row_stride;
        L.tile = simt_tile_index(*p);
        if (L.tile < 0) return fail(CBS_ERR_PLAN_MISMATCH, "unknown SIMT tile %dx%d", p->block_m, p->block_n);
        L.in_nhwc = d.in_layout == CBS_NHWC;
        L.out_nhwc = d.out_layout == CBS_NHWC;
        L.m_tiles = p->m_tiles; L.n_tiles = p->n_tiles;
        L.act = d.activation;
        L.residual = (const float *)residual;
        if (L.split > 1) {
            const size_t tiles = (size_t)p->m_tiles * p->n_tiles;
            const size_t counters = (tiles * sizeof(unsigned) + 255) / 256 * 256;
            L.counters = (unsigned int *)workspace;
            L.partials = (float *)((char *)workspace + counters);
        }
        return cuda_check(launch_simt(L, (cudaStream_t)stream), "SIMT kernel launch");
    }
    return launch_tc(*p, x, d.c_in_b > 0 ? x_b : nullptr, w_packed, bias, nullptr, 0.0f, residual, y, workspace,
                     (cudaStream_t)stream);
}

// Activation/residual agreement between a plan and the call's arguments.
cbs_status check_act_call(const cbs_plan_t *p, const void *residual) {
    if (p->desc.prec == CBS_INT8)
        return fail(CBS_ERR_INVALID_ARG, "INT8 plans run through cbs_conv_bn_silu_i8");
    if (p->desc.residual && !residual && p->desc.n > 0)
        return fail(CBS_ERR_INVALID_ARG, "residual is NULL for a plan with a residual");
    if (!p->desc.residual && residual)
        return fail(CBS_ERR_INVALID_ARG, "residual given for a plan without one");
    return CBS_OK;
}

}  // namespace

extern "C" {

cbs_status cbs_conv_bn_silu_f32(const cbs_plan_t *p, const void *x, const void *w_packed,
                                const float *bias, void *y, void *workspace, size_t workspace_bytes,
                                void *stream) {
    CBS_TRY(check_plan(p));
    if (p->desc.prec == CBS_INT8)
        return fail(CBS_ERR_INVALID_ARG, "INT8 plans run through cbs_conv_bn_silu_i8");
    if (p->desc.activation != CBS_ACT_SILU || p->desc.residual)
        return fail(CBS_ERR_INVALID_ARG, "plan asks for another activation or a residual: call cbs_conv_bn_act");
    if (p->desc.c_in_b > 0) return fail(CBS_ERR_INVALID_ARG, "two-input plan: call cbs_conv_bn_act_cat");
    return conv_act_impl(p, x, nullptr, w_packed, bias, nullptr, y, workspace, workspace_bytes, stream);
}

cbs_status cbs_conv_bn_act(const cbs_plan_t *p, const void *x, const void *w_packed, const float *bias,
                           const void *residual, void *y, void *workspace, size_t workspace_bytes, void *stream) {
    CBS_TRY(check_plan(p));
    CBS_TRY(check_act_call(p, residual));
    if (p->desc.c_in_b > 0) return fail(CBS_ERR_INVALID_ARG, "two-input plan: call cbs_conv_bn_act_cat");
    return conv_act_impl(p, x, nullptr, w_packed, bias, residual, y, workspace, workspace_bytes, stream);
}

cbs_status cbs_conv_bn_act_cat(const cbs_plan_t *p, const void *x, const void *x_b, const void *w_packed,
                               const float *bias, const void *residual, void *y, void *workspace,
                               size_t workspace_bytes, void *stream) {
    CBS_TRY(check_plan(p));
    CBS_TRY(check_act_call(p, residual));
    if (p->desc.c_in_b <= 0) return fail(CBS_ERR_INVALID_ARG, "one-input plan: call cbs_conv_bn_act");
    return conv_act_impl(p, x, x_b, w_packed, bias, residual, y, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// The INT8 layer, one or two inputs (checked against the plan by the caller).
cbs_status conv_i8_impl(const cbs_plan_t *p, const int8_t *x, const int8_t *x_b, const void *w_packed,
                        const int32_t *bias_i32, const float *m_c, float s_y, int8_t *y, void *workspace,
                        size_t workspace_bytes, void *stream) {
    if (p->desc.n == 0) return CBS_OK;  // empty batch: nothing is read or written
    CBS_TRY(check_conv_common(p, x, w_packed, bias_i32, y, workspace, workspace_bytes));
    if (p->desc.c_in_b > 0) CBS_TRY(check_ptr(x_b, "x_b"));
    CBS_TRY(check_ptr(m_c, "m_c"));
    if (!(s_y > 0.0f) || !(s_y < 3.0e38f)) return fail(CBS_ERR_INVALID_ARG, "s_y must be a positive finite float");
    const float inv_s_y = 1.0f / s_y;
    if (p->variant == CBS_VARIANT_STEM) {
        const StemLaunch L = stem_launch(*p, x, w_packed, bias_i32, m_c, inv_s_y, y);
        return cuda_check(launch_stem(L, (cudaStream_t)stream), "stem kernel launch");
    }
    return launch_tc(*p, x, p->desc.c_in_b > 0 ? x_b : nullptr, w_packed, bias_i32, m_c, inv_s_y, nullptr, y,
                     workspace, (cudaStream_t)stream);
}

}  // namespace

extern "C" {

cbs_status cbs_conv_bn_silu_i8(const cbs_plan_t *p, const int8_t *x, const void *w_packed,
                               const int32_t *bias_i32, const float *m_c, float s_y, int8_t *y,
                               void *workspace, size_t workspace_bytes, void *stream) {
    CBS_TRY(check_plan(p));
    if (p->desc.prec != CBS_INT8)
        return fail(CBS_ERR_INVALID_ARG, "plan is not an INT8 plan");
    if (p->desc.c_in_b > 0) return fail(CBS_ERR_INVALID_ARG, "two-input plan: call cbs_conv_bn_silu_i8_cat");
    return conv_i8_impl(p, x, nullptr, w_packed, bias_i32, m_c, s_y, y, workspace, workspace_bytes, stream);
}

cbs_status cbs_conv_bn_silu_i8_cat(const cbs_plan_t *p, const int8_t *x, const int8_t *x_b, const void *w_packed,
                                   const int32_t *bias_i32, const float *m_c, float s_y, int8_t *y,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    CBS_TRY(check_plan(p));
    if (p->desc.prec != CBS_INT8)
        return fail(CBS_ERR_INVALID_ARG, "plan is not an INT8 plan");
    if (p->desc.c_in_b <= 0) return fail(CBS_ERR_INVALID_ARG, "one-input plan: call cbs_conv_bn_silu_i8");
    return conv_i8_impl(p, x, x_b, w_packed, bias_i32, m_c, s_y, y, workspace, workspace_bytes, stream);
}

cbs_status cbs_maxpool2d(const void *x, void *y, int n, int c, int h, int w, int k, int stride, int pad,
                         int layout, int prec, void *stream) {
    CBS_TRY(check_ptr(x, "x"));
    CBS_TRY(check_ptr(y, "y"));
    if (n < 0 || c < 1 || h < 1 || w < 1 || k < 1 || stride < 1 || pad < 0 || 2 * pad > k || h + 2 * pad < k ||
        w + 2 * pad < k)
        return fail(CBS_ERR_INVALID_ARG, "bad max-pool shape (n=%d c=%d h=%d w=%d k=%d stride=%d pad=%d; pad <= k/2)",
                    n, c, h, w, k, stride, pad);
    if (layout != CBS_NCHW && layout != CBS_NHWC) return fail(CBS_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (prec < CBS_FP32 || prec > CBS_INT8) return fail(CBS_ERR_INVALID_ARG, "unknown precision %d", prec);
    if (n == 0) return CBS_OK;
    const int eb = prec == CBS_BF16 ? 2 : (prec == CBS_INT8 ? 1 : 4);
    return cuda_check(launch_maxpool(x, y, n, c, h, w, k, stride, pad, layout == CBS_NHWC, eb, (cudaStream_t)stream),
                      "max-pool launch");
}

cbs_status cbs_dequantize_i8(const int8_t *q, void *out, size_t count, float s, int z, int out_prec,
                             void *stream) {
    CBS_TRY(check_ptr(q, "q"));
    CBS_TRY(check_ptr(out, "out"));
    if (!(s > 0.0f) || !(s < 3.0e38f)) return fail(CBS_ERR_INVALID_ARG, "scale must be positive and finite");
    if (z < -128 || z > 127) return fail(CBS_ERR_INVALID_ARG, "zero point %d outside [-128, 127]", z);
    if (out_prec != CBS_FP32 && out_prec != CBS_TF32 && out_prec != CBS_BF16)
        return fail(CBS_ERR_INVALID_ARG, "output precision must be FP32, TF32 or BF16");
    if (count == 0) return CBS_OK;
    return cuda_check(launch_dequantize_i8(q, out, count, s, z, out_prec == CBS_BF16, (cudaStream_t)stream),
                      "dequantise launch");
}

cbs_status cbs_quantize_i8(const void *x, int in_prec, int8_t *q, size_t count, float s, int z, void *stream) {
    CBS_TRY(check_ptr(x, "x"));
    CBS_TRY(check_ptr(q, "q"));
    if (!(s > 0.0f) || !(s < 3.0e38f)) return fail(CBS_ERR_INVALID_ARG, "scale must be positive and finite");
    if (z < -128 || z > 127) return fail(CBS_ERR_INVALID_ARG, "zero point %d outside [-128, 127]", z);
    if (in_prec != CBS_FP32 && in_prec != CBS_TF32 && in_prec != CBS_BF16)
        return fail(CBS_ERR_INVALID_ARG, "input precision must be FP32, TF32 or BF16");
    if (count == 0) return CBS_OK;
    return cuda_check(launch_quantize_i8(x, in_prec == CBS_BF16, q, count, s, z, (cudaStream_t)stream),
                      "quantise launch");
}

cbs_status cbs_sppf_pool(const void *x, void *y, int n, int c, int h, int w, int k, int layout, int prec,
                         void *stream) {
    CBS_TRY(check_ptr(x, "x"));
    CBS_TRY(check_ptr(y, "y"));
    if (n < 0 || n > 65535 || c < 1 || h < 1 || w < 1 || k < 1 || k > 7 || !(k & 1))
        return fail(CBS_ERR_INVALID_ARG, "bad SPPF pool shape (n=%d c=%d h=%d w=%d k=%d; odd k <= 7)", n, c, h, w, k);
    if (layout != CBS_NCHW && layout != CBS_NHWC) return fail(CBS_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (prec < CBS_FP32 || prec > CBS_INT8) return fail(CBS_ERR_INVALID_ARG, "unknown precision %d", prec);
    if (n == 0) return CBS_OK;
    const int eb = prec == CBS_BF16 ? 2 : (prec == CBS_INT8 ? 1 : 4);
    return cuda_check(launch_sppf_pool(x, y, n, c, h, w, k, layout == CBS_NHWC, eb, (cudaStream_t)stream),
                      "SPPF pool launch");
}

cbs_status cbs_upsample2x_concat(const void *a, int ca, const void *b, int cb, void *out, int n, int h,
                                 int w, int layout, int elem_bytes, void *stream) {
    CBS_TRY(check_ptr(a, "a"));
    CBS_TRY(check_ptr(b, "b", cb == 0));
    CBS_TRY(check_ptr(out, "out"));
    if (ca < 1 || cb < 0 || n < 0 || h < 2 || w < 2 || (h & 1) || (w & 1))
        return fail(CBS_ERR_INVALID_ARG, "bad upsample/concat shape (ca=%d cb=%d n=%d h=%d w=%d; h, w even)",
                    ca, cb, n, h, w);
    if (layout != CBS_NCHW && layout != CBS_NHWC) return fail(CBS_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4)
        return fail(CBS_ERR_INVALID_ARG, "elem_bytes must be 1, 2 or 4 (got %d; ca=%d cb=%d n=%d h=%d w=%d layout=%d)",
                    elem_bytes, ca, cb, n, h, w, layout);
    if (n == 0) return CBS_OK;
    return cuda_check(launch_upsample_concat(a, ca, b, cb, out, n, h, w, layout == CBS_NHWC, elem_bytes,
                                             (cudaStream_t)stream),
                      "upsample/concat launch");
}

cbs_status cbs_workspace_init(void *workspace, size_t bytes, void *stream) {
    if (bytes == 0) return CBS_OK;
    CBS_TRY(check_ptr(workspace, "workspace"));
    return cuda_check(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream), "cudaMemsetAsync");
}

cbs_status cbs_read_device_status(int *status_out, int reset, void *stream) {
    if (!status_out) return fail(CBS_ERR_INVALID_ARG, "status_out is NULL");
    return read_and_reset_status(status_out, reset, (cudaStream_t)stream);
}

cbs_status cbs_selftest_wait_timeout(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 100000)
        return fail(CBS_ERR_INVALID_ARG, "limit_us %d: 1 .. 100000", limit_us);
    return cuda_check(launch_wait_selftest((unsigned long long)limit_us * 1000ull, (cudaStream_t)stream),
                      "wait self-test launch");
}

}  // extern "C"
