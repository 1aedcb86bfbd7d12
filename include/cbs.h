/*
 * cbs.h -- C ABI of the fused Conv2d + folded BatchNorm + SiLU library for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (page 1, "YOLO26N Inference Optimisation", sections
 * "NHWC migration -- What NHWC is and why it matters" and "Improvements",
 * #2 and #7; page 3, "Edge optimisation of YOLO26", "Design notes"):
 *
 *   y[n,co,oh,ow] = SiLU( sum_{r,s,ci} x[n, oh*S-P+r, ow*S-P+s, ci] * w'[co,r,s,ci] + b'[co] )
 *   w'[co,...] = w[co,...] * gamma[co] / sqrt(var[co] + eps)       (BN folded into the weights)
 *   b'[co]     = beta[co] - mean[co] * gamma[co] / sqrt(var[co] + eps)
 *   SiLU(z)    = z / (1 + exp(-z))
 *
 * x is zero outside the image.  Seen as a GEMM (page 1, "What NHWC is and why
 * it matters", item 3): A = [N*OH*OW, k*k*C_in] (the implicit im2col matrix),
 * B = [k*k*C_in, C_out].
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer unless the comment says host.
 *    The caller allocates and owns every buffer; the library never allocates,
 *    frees or synchronises device memory (except cbs_read_device_status,
 *    which synchronises the given stream by design).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All GPU work is enqueued on it and is asynchronous to the host.
 *  - Arguments are checked before anything is enqueued; on error nothing is
 *    enqueued and a status < 0 is returned.  cbs_last_error() then returns a
 *    message for the calling thread.
 *  - Device buffers must be 16-byte aligned (CBS_ERR_MISALIGNED otherwise).
 *  - All functions are re-entrant; message state is thread-local.
 */
#ifndef CBS_H
#define CBS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CBS_ABI_VERSION 5

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define CBS_API __attribute__((visibility("default")))
#else
#define CBS_API
#endif

typedef enum cbs_status {
    CBS_OK = 0,
    CBS_ERR_INVALID_ARG = -1,   /* bad shape, null pointer, unknown enum */
    CBS_ERR_UNSUPPORTED = -2,   /* valid but not implemented (e.g. layout for a variant) */
    CBS_ERR_MISALIGNED = -3,    /* a buffer is not 16-byte aligned */
    CBS_ERR_WORKSPACE = -4,     /* workspace missing or smaller than plan->workspace_bytes */
    CBS_ERR_CUDA = -5,          /* a CUDA runtime/driver call failed (launch, tensor map) */
    CBS_ERR_TIMEOUT = -6,       /* a bounded device-side wait expired (see cbs_read_device_status) */
    CBS_ERR_PLAN_MISMATCH = -7  /* plan is not a plan of this library version */
} cbs_status;

/* Activation layouts (page 1, "What must change in the kernels"). */
typedef enum cbs_layout { CBS_NCHW = 0, CBS_NHWC = 1 } cbs_layout;

/* Arithmetic variant.  Storage type of x and y: FP32 and TF32 use float,
 * BF16 uses bfloat16, INT8 uses int8.  Accumulation: float (FP32 FMA on CUDA
 * cores; TF32/BF16 tensor cores), exact integer for INT8. */
typedef enum cbs_precision { CBS_FP32 = 0, CBS_TF32 = 1, CBS_BF16 = 2, CBS_INT8 = 3 } cbs_precision;

/* Activation after the folded BatchNorm.  SiLU is the fused layer of the
 * pages; identity gives the plain convolution + bias that page 1's kernel
 * profile also runs ("conv2d_forward").  FP32, TF32 and BF16 only. */
typedef enum cbs_activation { CBS_ACT_SILU = 0, CBS_ACT_IDENTITY = 1 } cbs_activation;

/* Kernel family a plan selects. */
typedef enum cbs_variant {
    CBS_VARIANT_SIMT_FP32 = 0,  /* CUDA-core implicit GEMM, FP32 FMA */
    CBS_VARIANT_TC_TF32 = 1,    /* tcgen05 kind::tf32, TMA im2col/tile loads, TMEM accumulator */
    CBS_VARIANT_TC_BF16 = 2,    /* tcgen05 kind::f16 (bf16 operands) */
    CBS_VARIANT_TC_INT8 = 3,    /* int8 values on tcgen05 kind::f16, exact integer sums */
    CBS_VARIANT_STEM = 4,       /* direct CUDA-core convolution for C_in <= 4 (any precision) */
    CBS_VARIANT_TC_TF32X3 = 5   /* FP32 on tcgen05 kind::tf32: operands split into a TF32 head and a tail,
                                   three MMAs per K slice (head x head + head x tail + tail x head) */
} cbs_variant;

/* One layer.  Padding is symmetric; OH = (H + 2*pad - k)/stride + 1. */
typedef struct cbs_layer_desc {
    int n, c_in, h, w, c_out, k, stride, pad;
    int in_layout;       /* cbs_layout of x */
    int out_layout;      /* cbs_layout of y */
    int prec;            /* cbs_precision */
    int force_variant;   /* -1: choose from prec; else a cbs_variant compatible with prec */
    int force_split_k;   /* 0: choose; else the number of K splits to use (>= 1).  Tensor-core
                            variants (TF32/BF16): on request only, with im2col or 2-D A and
                            streamed weights; the plan then needs a workspace */
    int force_block_n;   /* 0: choose; else the N tile width (must be one the variant supports) */
    int force_block_m;   /* 0: choose; else the M tile height (CUDA-core variant: 64, 128 or 256;
                            TF32/BF16 tensor-core variants: 128 or 256) */
    int out_row_stride;  /* NCHW output only: elements between output rows; 0 = OW.
                            Must be >= OW.  Columns OW..stride-1 are never written. */
    int force_k_group;   /* TF32/BF16: 0 = choose; else K steps per pipeline stage (divides the
                            layer's K steps) */
    int force_b_resident;/* TF32/BF16: 0 = choose; 1 = keep weights resident in shared memory;
                            -1 = stream them with every K step */
    int force_window;    /* TF32/BF16: 1 = windowed A (stride 1, odd k, pad k/2, channel blocks of
                            128 bytes); 0 or -1 = im2col A.
                            TF32X3 with NCHW input: 1 = flat input boxes (stride 1, k = 2 pad + 1
                            <= 7, W a multiple of 4, and N = 1 or OH*OW a multiple of 128;
                            CBS_ERR_UNSUPPORTED otherwise); 0 or -1 = the converter warps load the
                            input themselves.  TF32X3 with NHWC input: must not be 1.  The
                            CUDA-core, stem and INT8 variants ignore it. */
    int activation;      /* cbs_activation (0 = SiLU) */
    int residual;        /* 1: add a residual tensor to the activated output, y = act(z) + r
                            (page 1's profile: the element-wise adds beside the convolutions);
                            the layer is then called through cbs_conv_bn_act.  FP32/TF32/BF16. */
    int c_in_b;          /* 0: one input tensor x.  > 0: the layer's input is the channel
                            concatenation of two tensors (page 1, "Improvements" #6, channel_cat
                            fused into the convolution's input loads): channels 0..c_in-c_in_b-1
                            come from x and the last c_in_b from x_b, both with the same N, H, W
                            and layout; the layer is then called through cbs_conv_bn_act_cat.
                            FP32 (CUDA-core variant), TF32, BF16 and INT8 (both inputs with the
                            same scale and zero point; called through cbs_conv_bn_silu_i8_cat);
                            the tensor-core variants need c_in - c_in_b to be a multiple of 16
                            (BF16, INT8) or 8 (TF32) channels and c_in_b a multiple of 16 (INT8),
                            8 (BF16) or 4 (TF32). */
    int zero_point_x;    /* INT8: zero point z_x in [-128, 127] of the input codes (asymmetric
                            activations, page 3 "Design notes": a code q stands for s_x (q - z_x);
                            a uint8 code u with zero point z_u is q = u - 128, z_x = z_u - 128).
                            0 = symmetric.  Must be 0 for the other precisions. */
    int zero_point_y;    /* INT8: zero point z_y in [-128, 127] of the output codes. */
    int num_sms;         /* SMs of the device the layer will run on (cudaDevAttrMultiProcessorCount):
                            grids, waves and split-K are sized for it.  0 = 152, the GB300's count.
                            cbs_plan stays a pure host function: it never queries the device. */
    int force_issuer_split; /* TF32/BF16: 1 = the K stages of each 128-pixel tile alternate
                            between the kernel's two MMA-issuing threads, each summing into an
                            accumulator of its own that the epilogue adds (needs block_m 128,
                            im2col A, no split-K, at least two stages per tile and an N tile of
                            at most 128); 0 or -1 = one issuing thread per 128-pixel tile.  On
                            request only: measured slower than the planner's choice on most
                            layers.  Must be 0 or -1 for the other variants. */
} cbs_layer_desc;

/* A plan: plain data, owned by the caller, filled by cbs_plan. */
typedef struct cbs_plan_t {
    uint32_t size;          /* sizeof(cbs_plan_t); checked by every call */
    uint32_t abi_version;   /* CBS_ABI_VERSION */
    int variant;            /* cbs_variant */
    int block_m, block_n, block_k;  /* CTA tile: output pixels x output channels x K step */
    int stages;             /* shared-memory pipeline depth */
    int split_k;            /* number of K partitions (>= 1) */
    int k_group;            /* tensor-core variants: K steps carried by one pipeline stage
                               (windowed plans: slots of the weight ring, 0 if resident) */
    int b_resident;         /* tensor-core variants: 1 = each CTA loads its weight tile once
                               and keeps it in shared memory for the whole launch */
    int window;             /* TF32/BF16, stride 1: 1 = each tile loads its zero-padded input
                               window once per channel block and every filter tap reads a
                               shifted view of it (block_m positions of the padded grid
                               oh * (W + 2 pad) + ow'); 0 = one im2col box per tap.
                               TF32X3 with NCHW input: 1 = each K step's input arrives as one
                               TMA box of 136 pixels of a filter row's flat H*W channel rows
                               (the converter warps zero the columns that wrap); 0 = the
                               converter warps load it from global memory */
    int issuer_split;       /* TF32/BF16: 2 = each 128-pixel tile's K stages alternate between
                               two MMA-issuing threads (see force_issuer_split); else 1 */
    int c_in_pad;           /* channels per input pixel as stored (NHWC tensor-core variants
                               pad C_in to a 16-byte multiple; SIMT: = c_in) */
    int k_gemm;             /* GEMM K = k*k*c_in_pad: length of one packed weight row */
    int oh, ow;
    int out_row_stride;     /* NCHW: elements between output rows (>= ow) */
    int m_tiles, n_tiles;   /* tile grid */
    int grid_ctas;          /* CTAs launched */
    int threads;            /* threads per CTA */
    int smem_bytes;         /* dynamic shared memory per CTA */
    size_t x_bytes;         /* bytes of x the kernel reads, in the plan's input format */
    size_t y_bytes;         /* bytes of y, including row padding */
    size_t w_packed_bytes;  /* bytes of the packed weight buffer */
    size_t bias_bytes;      /* bytes of the bias buffer (float or int32 per channel) */
    size_t workspace_bytes; /* scratch the call needs (0 = none) */
    size_t x_b_bytes;       /* two-input plans: bytes of x_b the kernel reads (x_bytes is then
                               x's share); 0 for one-input plans */
    cbs_layer_desc desc;    /* copy of the request */
} cbs_plan_t;

/*
 * cbs_plan -- choose a kernel variant and tile configuration for one layer
 * (page 1, "Key observations" 1 and "Improvements" #1: one tile configuration
 * per call-site shape instead of one for all 40 convolutions).
 *   d:   host pointer to the layer; out: host pointer, filled on success.
 * Host only: makes no CUDA call and may be used without a GPU.
 * Variant choice (force_variant = -1): STEM for the small-channel stems
 * below; else the precision's own variant, except that an FP32 layer takes
 * TC_TF32X3 (the FP32 bar on the tensor cores, split-K where its tiles leave
 * SMs idle) when each input's channel count is a multiple of 8, no tile
 * field is forced, and either its input is NHWC or it is a one-input layer
 * with NCHW input, k >= 3 and stride 1; it falls back to SIMT FP32 when no
 * 3xTF32 configuration fits.  Its input is then the same bytes as for SIMT
 * FP32.
 * Input format the plan expects (see x_bytes):
 *   SIMT FP32: x in d->in_layout, float, exactly C_in channels.
 *   TF32/BF16/INT8 and TF32X3 (FP32): x NHWC with c_in_pad channels (extra
 *   channels zero; TF32X3: c_in_pad = C_in rounded up to 8).
 *   TF32X3 with NCHW input (one input only): x NCHW float, exactly C_in
 *   channels, read as given by the kernel.
 *   STEM (chosen for C_in <= 4, C_out <= 64, k <= 7): x in d->in_layout;
 *   NHWC pixels hold c_in_pad = 4 channels for TF32/BF16/INT8, C_in for FP32.
 *   Two-input plans (d->c_in_b > 0): x holds the first c_in - c_in_b channels
 *   exactly; x_b the other c_in_b (SIMT FP32) or c_in_pad - (c_in - c_in_b)
 *   (TF32/BF16, extra channels zero).
 * Errors: CBS_ERR_INVALID_ARG (shape, enum), CBS_ERR_UNSUPPORTED.
 */
CBS_API cbs_status cbs_plan(const cbs_layer_desc *d, cbs_plan_t *out);

/*
 * cbs_fold_bn -- one-time weight transform (page 1, "Weight layout";
 * "Improvements" #7; page 3, "Design notes", per-channel weights).
 * Folds inference BatchNorm into the weights and bias, re-lays the weights
 * from [C_out][C_in][k][k] to the variant's K-major packed form with k-order
 * (r, s, ci), and casts or quantises them:
 *   SIMT FP32: float  [k*k*C_in][C_out]
 *   TF32, STEM with FP32/TF32: float [C_out][k*k*c_in_pad] (padding channels zero)
 *   TF32X3:    float [2*C_out][k*k*c_in_pad]: rows 0..C_out-1 the heads (w' with
 *              its low 13 mantissa bits cleared), rows C_out.. the tails w' - head
 *   BF16:      bf16   [C_out][k*k*c_in_pad]   (round to nearest even)
 *   INT8:      int8 codes held exactly as bf16 [C_out][k*k*c_in_pad];
 *              s_w[c] = max|w'[c,:]| / 127, q = rne(w'/s_w), m_c[c] = s_x * s_w[c],
 *              bias_i32[c] = rne(b'[c] / m_c[c]) saturated.  With an input zero
 *              point z_x != 0 the bias written is bias_i32[c] - z_x * sum q[c, :]
 *              (two's-complement int32): the kernels read the code z_x (a real
 *              zero) for every tap outside the image.
 * Arguments (device): w_oihw float[C_out*C_in*k*k]; conv_bias float[C_out] or
 * NULL; gamma, beta, mean, var float[C_out]; eps > 0.  s_x: activation scale
 * (INT8 only, else ignored).  Outputs: w_packed (plan->w_packed_bytes), bias
 * (float[C_out], or int32[C_out] for INT8), m_c (float[C_out], INT8 only,
 * may be NULL otherwise).  The float arithmetic uses fixed IEEE operations
 * (no contraction), so the INT8 codes are reproducible bit for bit.
 */
CBS_API cbs_status cbs_fold_bn(const cbs_plan_t *p, const float *w_oihw, const float *conv_bias,
                       const float *gamma, const float *beta, const float *mean,
                       const float *var, float eps, float s_x,
                       void *w_packed, void *bias, float *m_c, void *stream);

/*
 * cbs_pack_input -- chain-entry layout step (page 1, "The all-or-nothing
 * constraint", item 1: one NCHW->NHWC conversion at graph entry).
 * x_nchw: float [N][C_in][H][W].  x_packed: the plan's input format
 * (plan->x_bytes): SIMT with NCHW input: a copy; SIMT with NHWC input: float
 * NHWC; TF32: float NHWC padded to c_in_pad with zeros; BF16: bf16 (RNE);
 * INT8: int8 q = clamp(rne(x / s_x) + z_x, -128, 127) with the plan's zero
 * point z_x (0: symmetric); padding channels hold code 0.  Two-input plans:
 * CBS_ERR_UNSUPPORTED (each input is an earlier layer's output, or is packed
 * with a one-input plan of its own channel count).
 */
CBS_API cbs_status cbs_pack_input(const cbs_plan_t *p, const float *x_nchw, void *x_packed, float s_x,
                          void *stream);

/*
 * cbs_conv_bn_silu_f32 -- the fused layer for the FP32, TF32 and BF16
 * variants.  x: plan input format; w_packed, bias: from cbs_fold_bn; y: output
 * in d.out_layout, float for FP32/TF32, bf16 for BF16 (plan->y_bytes);
 * workspace: plan->workspace_bytes bytes (may be NULL when that is 0) which
 * must have been zeroed once with cbs_workspace_init before its first use;
 * every call leaves it ready for the next one.  A workspace must not be
 * shared by calls that may run concurrently.
 */
CBS_API cbs_status cbs_conv_bn_silu_f32(const cbs_plan_t *p, const void *x, const void *w_packed,
                                const float *bias, void *y, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * cbs_conv_bn_act -- the same layer with the descriptor's activation and an
 * optional residual add, fused into the epilogue:
 *   y = act(conv(x) * s + b') + r
 * (the residual and plain-bias forms of page 1's kernel profile:
 * "conv2d_forward", "elemwise_add").  residual: device pointer, NULL unless
 * p->desc.residual; same layout, element type and row pitch as y.  It may be
 * y itself (in-place add).  Other arguments, ownership and errors as for
 * cbs_conv_bn_silu_f32, which accepts only SiLU plans without a residual.
 * CBS_ERR_INVALID_ARG if residual is NULL for a residual plan, or non-NULL
 * for one without.
 */
CBS_API cbs_status cbs_conv_bn_act(const cbs_plan_t *p, const void *x, const void *w_packed, const float *bias,
                                   const void *residual, void *y, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * cbs_conv_bn_act_cat -- cbs_conv_bn_act for a two-input plan (d.c_in_b > 0):
 * the convolution's input is concat(x, x_b) along channels, read straight from
 * the two tensors (no concatenated copy is made).  x: the plan's input format
 * with c_in - c_in_b channels; x_b: the same format with the remaining
 * channels (see cbs_plan).  Other arguments, ownership and errors as for
 * cbs_conv_bn_act.  The one-input entry points reject two-input plans
 * (CBS_ERR_INVALID_ARG), and this one rejects one-input plans.
 */
CBS_API cbs_status cbs_conv_bn_act_cat(const cbs_plan_t *p, const void *x, const void *x_b, const void *w_packed,
                                       const float *bias, const void *residual, void *y, void *workspace,
                                       size_t workspace_bytes, void *stream);

/*
 * cbs_conv_bn_silu_i8 -- the fused INT8 layer (page 3, "Highlights" and
 * "Design notes": per-output-channel weight scales, one activation scale).
 *   acc   = sum over the taps inside the image of (q_x - z_x) * q_w
 *           + bias_i32                        (exact integer; z_x = 0: symmetric)
 *   t     = float(acc) * m_c[co]
 *   u     = t / (1 + e(-t))                   (SiLU in float; e = the library's
 *                                              Cody-Waite/Taylor exp, bit-specified)
 *   q_y   = clamp(rne(u * (1/s_y)) + z_y, -128, 127)
 * z_x, z_y: the plan's zero points.  w_packed and bias_i32 as written by
 * cbs_fold_bn for this plan.
 * x: int8 NHWC with c_in_pad channels; y: int8 in d.out_layout.
 * Workspace rules as for cbs_conv_bn_silu_f32.
 */
CBS_API cbs_status cbs_conv_bn_silu_i8(const cbs_plan_t *p, const int8_t *x, const void *w_packed,
                               const int32_t *bias_i32, const float *m_c, float s_y,
                               int8_t *y, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * cbs_conv_bn_silu_i8_cat -- cbs_conv_bn_silu_i8 for a two-input plan: the
 * input is concat(x, x_b) along channels, read straight from the two int8
 * tensors (same scale s_x and zero point z_x).  x: NHWC int8 with
 * c_in - c_in_b channels; x_b: NHWC int8 with c_in_pad - (c_in - c_in_b)
 * channels (extra channels 0).  Other arguments and errors as for
 * cbs_conv_bn_silu_i8, which rejects two-input plans (and this one-input ones).
 */
CBS_API cbs_status cbs_conv_bn_silu_i8_cat(const cbs_plan_t *p, const int8_t *x, const int8_t *x_b,
                                           const void *w_packed, const int32_t *bias_i32, const float *m_c,
                                           float s_y, int8_t *y, void *workspace, size_t workspace_bytes,
                                           void *stream);

/*
 * cbs_upsample2x_concat -- neck glue between two fused layers (page 1,
 * "Op-by-op impact", upsample_nearest2d and channel_cat):
 *   out[n, h, w, :] = concat( a[n, h/2, w/2, 0:ca], b[n, h, w, 0:cb] )
 * layout: CBS_NHWC or CBS_NCHW for all three tensors; elem_bytes: 1, 2 or 4.
 * a: [n][h/2][w/2][ca]; b, out: [n][h][w][cb] and [n][h][w][ca+cb] (as NHWC).
 * cb = 0 (b may then be NULL) gives the plain nearest 2x upsample of a, the
 * form that feeds a two-input layer (cbs_conv_bn_act_cat) directly.
 */
CBS_API cbs_status cbs_upsample2x_concat(const void *a, int ca, const void *b, int cb, void *out,
                                 int n, int h, int w, int layout, int elem_bytes,
                                 void *stream);

/*
 * cbs_maxpool2d -- max pooling beside the convolutions (page 1, "YOLO26N
 * Inference Optimisation", kernel profile and "Op-by-op impact": maxpool2d,
 * the SPPF block's 5x5 stride-1 pools):
 *   y[n,c,oh,ow] = max of x over the k x k window at (oh*stride-pad,
 *                  ow*stride-pad), positions outside the image taking no part
 * OH = (h + 2 pad - k)/stride + 1 (floor), likewise OW; 0 <= pad <= k/2.  A
 * NaN in the window gives NaN.  x: [n][c][h][w] (NCHW) or [n][h][w][c]
 * (NHWC); y the same layout with OH x OW.  prec: the element type as for a
 * layer (FP32/TF32 float, BF16 bfloat16, INT8 int8 codes, which compare like
 * their values).  Errors: CBS_ERR_INVALID_ARG for shapes and enums.
 */
CBS_API cbs_status cbs_maxpool2d(const void *x, void *y, int n, int c, int h, int w, int k, int stride, int pad,
                                 int layout, int prec, void *stream);

/*
 * cbs_dequantize_i8, cbs_quantize_i8 -- the seams between INT8 layers and
 * layers kept in float (page 3, "Edge optimisation of YOLO26", "Highlights":
 * a layer-sensitivity analysis keeps some layers in float), in the affine
 * scheme r = s (q - z) of the INT8 path:
 *   dequantise: out[i] = (float)(q[i] - z) * s    (one IEEE multiply; BF16
 *               output rounded to nearest even)
 *   quantise:   q[i] = clamp(rne(x[i] / s) + z, -128, 127)   (IEEE division;
 *               the quantiser of cbs_pack_input)
 * count values, elementwise, any layout (NHWC activations whose channel
 * counts are the same in both formats).  out_prec / in_prec: CBS_FP32 or
 * CBS_TF32 (float), or CBS_BF16 (bfloat16).  s > 0, z in [-128, 127].
 * Errors: CBS_ERR_INVALID_ARG, CBS_ERR_MISALIGNED (16-byte alignment).
 */
CBS_API cbs_status cbs_dequantize_i8(const int8_t *q, void *out, size_t count, float s, int z, int out_prec,
                                     void *stream);
CBS_API cbs_status cbs_quantize_i8(const void *x, int in_prec, int8_t *q, size_t count, float s, int z,
                                   void *stream);

/*
 * cbs_sppf_pool -- the SPPF block's three chained max pools in one launch
 * (page 1, "YOLO26N Inference Optimisation", kernel profile and "Op-by-op
 * impact": maxpool2d, three per frame, each a 5x5 stride-1 pool feeding the
 * next, their outputs concatenated with the pools' input):
 *   y = concat(p(x), p(p(x)), p(p(p(x))))   along channels,
 *   p = the k x k max pool with stride 1 and padding k/2, positions outside
 *       the image taking no part (cbs_maxpool2d with stride 1, pad k/2).
 * The result is the same, bit for bit, as three cbs_maxpool2d calls.  The
 * fourth part of the block's concatenation, x itself, is not copied: the next
 * layer reads concat(x, y) through a two-input plan (c_in_b = 3c).
 * x: [n][c][h][w] (NCHW) or [n][h][w][c] (NHWC); y: [n][3c][h][w] or
 * [n][h][w][3c].  k odd, 1..7.  prec: element type as for cbs_maxpool2d.
 * A NaN in a window gives NaN.  Errors: CBS_ERR_INVALID_ARG for shapes and
 * enums (n <= 65535).
 */
CBS_API cbs_status cbs_sppf_pool(const void *x, void *y, int n, int c, int h, int w, int k, int layout, int prec,
                                 void *stream);

/*
 * cbs_conv_bn_silu_f32_noalloc -- the FP32 CUDA-core fused layer for callers
 * that cannot allocate device memory.  No passage of the pages has a
 * counterpart: this is a deployment interface, not part of the method.
 * Some callers hold only the layer's own buffers: a plugin interface that
 * passes input and output pointers and no workspace, or a latency-bound
 * serving loop that must not allocate after start-up (cudaMalloc can
 * synchronise the device).  This call needs no workspace argument: split-K
 * scratch comes from a 16 MiB array the library defines in device memory
 * (present on every GPU that loads the library, until the process exits).
 *   p: a CBS_VARIANT_SIMT_FP32 plan with workspace_bytes <= 16 MiB (larger
 *      plans fail with CBS_ERR_WORKSPACE; other variants CBS_ERR_UNSUPPORTED).
 *      An FP32 layer with NHWC input plans TC_TF32X3 by default: set
 *      force_variant = CBS_VARIANT_SIMT_FP32 in its descriptor for this call;
 *   x, w_packed, bias, y: as for cbs_conv_bn_silu_f32 (device, 16-byte aligned).
 * The first call on a device looks up the array's address with that device
 * current; make it before any stream capture.  Every call shares the array
 * and zeroes its split-K counters on `stream` before its kernel; calls whose
 * kernels may overlap on the GPU race on the array and give wrong results.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
CBS_API cbs_status cbs_conv_bn_silu_f32_noalloc(const cbs_plan_t *p, const float *x, const float *w_packed,
                                                const float *bias, float *y, void *stream);

/*
 * cbs_set_launch_options -- process-wide launch options for every kernel
 * the library enqueues afterwards (a bit set, CBS_LAUNCH_*):
 *   CBS_LAUNCH_PDL  programmatic dependent launch (default on) of the
 *                   tensor-core kernels, the tensor-core stem and the
 *                   packing and glue kernels: a kernel may be scheduled while
 *                   the previous kernel in the stream finishes, runs its
 *                   set-up (barriers, tensor memory, tensor-map prefetch)
 *                   meanwhile, and waits for that kernel before it reads or
 *                   writes global memory.  The CUDA-core kernels always use
 *                   plain launches (measured faster).  Results are the same
 *                   with the bit clear; only the gap between kernels changes.
 *                   Inside a CUDA graph capture the dependency becomes a
 *                   programmatic edge.
 * Not synchronised with launches in flight on other threads.
 * Errors: CBS_ERR_INVALID_ARG for unknown bits.
 */
#define CBS_LAUNCH_PDL 1
CBS_API cbs_status cbs_set_launch_options(int flags);
CBS_API int cbs_launch_options(void);

/* Zero a workspace before its first use (cudaMemsetAsync on `stream`). */
CBS_API cbs_status cbs_workspace_init(void *workspace, size_t bytes, void *stream);

/*
 * cbs_read_device_status -- synchronise `stream`, then report whether any
 * kernel of this library on the current device gave up a bounded wait since
 * the last reset: *status_out (host) receives CBS_OK or CBS_ERR_TIMEOUT.
 * reset != 0 clears the flag.
 */
CBS_API cbs_status cbs_read_device_status(int *status_out, int reset, void *stream);

/*
 * cbs_selftest_wait_timeout -- diagnostic of the timeout path (no passage of
 * the pages has a counterpart).  Enqueues one CTA on `stream` whose thread
 * waits, through the same bounded mbarrier wait the tensor-core kernels use,
 * on a barrier that nothing arrives at.  After limit_us microseconds
 * (1 .. 100000) the wait gives up and the kernel records a timeout in the
 * status word, exactly as a layer kernel does when one of its waits runs
 * out; cbs_read_device_status then reports CBS_ERR_TIMEOUT.  Nothing faults
 * and the context stays usable.  Errors: CBS_ERR_INVALID_ARG for limit_us
 * out of range, CBS_ERR_CUDA if the launch fails.
 */
CBS_API cbs_status cbs_selftest_wait_timeout(int limit_us, void *stream);

/* Static string for a status code. */
CBS_API const char *cbs_status_string(cbs_status s);

/* Message for the last failing call on this thread ("" if none). */
CBS_API const char *cbs_last_error(void);

/* CBS_ABI_VERSION of the loaded library. */
CBS_API int cbs_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CBS_H */
