"""Host-side checks of the C ABI: the library loads without a GPU, exports
every function include/cbs.h declares, and its planner and argument checks
behave as documented (none of these calls reach the GPU)."""
import ctypes
import os
import re

import pytest

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import make_desc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "cbs.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CBS_API\s+[\w\s\*]+?\b(cbs_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(cuda_lib):
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(cuda_lib, name), name
    assert set(names) == set(B.EXPORTED)


def test_abi_version_and_struct_sizes(cuda_lib):
    assert B.cbs_abi_version() == 5
    plan = B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1))
    assert plan.size == ctypes.sizeof(B.cbs_plan_t)
    assert plan.abi_version == 5


def test_status_strings(cuda_lib):
    for code, name in [(0, "CBS_OK"), (-1, "CBS_ERR_INVALID_ARG"), (-2, "CBS_ERR_UNSUPPORTED"),
                       (-3, "CBS_ERR_MISALIGNED"), (-4, "CBS_ERR_WORKSPACE"), (-5, "CBS_ERR_CUDA"),
                       (-6, "CBS_ERR_TIMEOUT"), (-7, "CBS_ERR_PLAN_MISMATCH")]:
        assert B.cbs_status_string(code) == name


@pytest.mark.parametrize("i", range(len(wl.LAYER_LIST)))
def test_plan_fp32_layer_list(cuda_lib, i):
    s = wl.LAYER_LIST[i]
    p = B.cbs_plan(make_desc(1, s.c_in, s.h, s.width, s.c_out, s.k, s.stride))
    # Three-channel stems take the direct CUDA-core kernel; layers with 32 or
    # more channels and a 3x3 filter, or 64 or more channels, the 3xTF32
    # tensor-core kernel (reading the NCHW input as given); the rest the
    # CUDA-core implicit GEMM.
    x3 = s.c_in >= 32 and (s.k == 3 or s.c_in >= 64)
    assert p.variant == (B.CBS_VARIANT_STEM if s.c_in <= 4 else
                         B.CBS_VARIANT_TC_TF32X3 if x3 else B.CBS_VARIANT_SIMT_FP32)
    assert (p.oh, p.ow) == (s.oh, s.ow)
    assert p.out_row_stride == s.ow
    assert p.x_bytes == s.c_in * s.h * s.width * 4
    assert p.y_bytes == s.c_out * s.oh * s.ow * 4
    # (3xTF32 keeps each weight as a TF32 head and the remainder)
    assert p.w_packed_bytes == s.c_out * s.c_in * s.k * s.k * 4 * (2 if x3 else 1)
    assert p.m_tiles * p.block_m >= s.oh * s.ow
    assert p.n_tiles * p.block_n >= s.c_out
    if x3:
        assert p.grid_ctas <= 152 and (p.workspace_bytes > 0) == (p.split_k > 1)
    else:
        assert p.split_k >= 1 and p.grid_ctas == p.m_tiles * p.n_tiles * p.split_k
        assert (p.workspace_bytes > 0) == (p.split_k > 1)


def test_fp32_nchw_tensor_core_rules(cuda_lib):
    """NCHW FP32 layers go to the 3xTF32 kernel when C_in is a multiple of 8,
    at least 32, and either k >= 3 or C_in >= 64, with nothing forced;
    forcing the variant takes any one-input NCHW layer there; a two-input
    NCHW layer cannot."""
    X3 = B.CBS_VARIANT_TC_TF32X3
    auto = lambda **kw: B.cbs_plan(make_desc(**dict(dict(n=1, c_in=64, h=20, w=20, c_out=64, k=3, stride=1), **kw)))
    assert auto().variant == X3
    assert auto(stride=2).variant == X3
    assert auto(k=1).variant == X3
    assert auto(k=1, c_in=32).variant == B.CBS_VARIANT_SIMT_FP32
    assert auto(c_in=32).variant == X3
    assert auto(c_in=16).variant == B.CBS_VARIANT_SIMT_FP32
    assert auto(c_in=60).variant == B.CBS_VARIANT_SIMT_FP32
    assert auto(force_block_m=64).variant == B.CBS_VARIANT_SIMT_FP32        # a forced tile is the CUDA-core kernel's
    forced = auto(k=1, c_in=20, force_variant=X3)
    assert forced.variant == X3 and forced.c_in_pad == 24 and forced.x_bytes == 20 * 20 * 20 * 4
    with pytest.raises(B.CbsError) as e:
        auto(c_in_b=32, force_variant=X3)
    assert e.value.status == B.CBS_ERR_UNSUPPORTED


def test_plan_stem_rules(cuda_lib):
    for prec, c_pad in ((B.CBS_FP32, 3), (B.CBS_TF32, 4), (B.CBS_BF16, 4), (B.CBS_INT8, 4)):
        p = B.cbs_plan(make_desc(2, 3, 64, 64, 16, 3, 2, prec=prec, in_layout=B.CBS_NHWC))
        assert p.variant == B.CBS_VARIANT_STEM and p.c_in_pad == c_pad
    # forcing the implicit GEMM for a small-channel FP32 layer stays possible
    p = B.cbs_plan(make_desc(1, 3, 64, 64, 16, 3, 2, force_variant=B.CBS_VARIANT_SIMT_FP32))
    assert p.variant == B.CBS_VARIANT_SIMT_FP32
    with pytest.raises(B.CbsError) as e:
        B.cbs_plan(make_desc(1, 8, 64, 64, 16, 3, 2, force_variant=B.CBS_VARIANT_STEM))
    assert e.value.status == B.CBS_ERR_UNSUPPORTED


def test_plan_padded_row_stride(cuda_lib):
    p = B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1, out_row_stride=48))
    assert p.out_row_stride == 48 and p.y_bytes == 32 * 40 * 48 * 4


def test_plan_forced_split(cuda_lib):
    for split in (1, 2, 5, 9):
        p = B.cbs_plan(make_desc(1, 256, 20, 20, 256, 3, 1, force_split_k=split))
        assert p.split_k == split


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), B.CBS_ERR_INVALID_ARG),
    (dict(c_in=0), B.CBS_ERR_INVALID_ARG),
    (dict(pad=3), B.CBS_ERR_UNSUPPORTED),
    (dict(prec=7), B.CBS_ERR_INVALID_ARG),
    (dict(out_row_stride=39), B.CBS_ERR_INVALID_ARG),
    (dict(out_row_stride=48, out_layout=B.CBS_NHWC), B.CBS_ERR_INVALID_ARG),
    (dict(force_variant=2), B.CBS_ERR_INVALID_ARG),
    (dict(in_layout=5), B.CBS_ERR_INVALID_ARG),
    (dict(h=1, w=1, pad=0), B.CBS_ERR_INVALID_ARG),
])
def test_plan_rejects(cuda_lib, kw, status):
    args = dict(n=1, c_in=16, h=40, w=40, c_out=32, k=3, stride=1, pad=1)
    args.update(kw)
    with pytest.raises(B.CbsError) as e:
        B.cbs_plan(make_desc(**args))
    assert e.value.status == status


def test_call_checks_before_any_launch(cuda_lib):
    """Argument errors are reported without touching the GPU."""
    p = B.cbs_plan(make_desc(1, 256, 20, 20, 256, 3, 1, force_split_k=4))
    ok = 1 << 20
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32(p, None, ok, ok, ok, ok, p.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32(p, ok + 4, ok, ok, ok, ok, p.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_MISALIGNED
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32(p, ok, ok, ok, ok, None, 0, None)
    assert e.value.status == B.CBS_ERR_WORKSPACE
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32(p, ok, ok, ok, ok, ok, p.workspace_bytes - 1, None)
    assert e.value.status == B.CBS_ERR_WORKSPACE
    bad = B.cbs_plan_t.from_buffer_copy(p)
    bad.size = 3
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32(bad, ok, ok, ok, ok, ok, p.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_PLAN_MISMATCH
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_i8(p, ok, ok, ok, ok, 0.1, ok, ok, p.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_upsample2x_concat(ok, 4, ok, 4, ok, 1, 5, 4, B.CBS_NHWC, 2, None)
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    assert "odd" in B.cbs_last_error() or "shape" in B.cbs_last_error()


def test_activation_and_residual_argument_rules(cuda_lib):
    """Host-side checks of the activation / residual plans (no launch)."""
    ok = 1 << 20
    with pytest.raises(B.CbsError) as e:
        B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1, activation=2))
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    for kw in (dict(activation=B.CBS_ACT_IDENTITY), dict(residual=1)):
        with pytest.raises(B.CbsError) as e:
            B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1, prec=B.CBS_INT8, in_layout=B.CBS_NHWC, **kw))
        assert e.value.status == B.CBS_ERR_UNSUPPORTED
    ident = B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1, activation=B.CBS_ACT_IDENTITY))
    resid = B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1, residual=1))
    plain = B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1))
    for p in (ident, resid):   # the SiLU entry point refuses them
        with pytest.raises(B.CbsError) as e:
            B.cbs_conv_bn_silu_f32(p, ok, ok, ok, ok, ok, p.workspace_bytes, None)
        assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_act(resid, ok, ok, ok, None, ok, ok, resid.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_act(plain, ok, ok, ok, ok, ok, ok, plain.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_act(resid, ok, ok, ok, ok + 8, ok, ok, resid.workspace_bytes, None)
    assert e.value.status == B.CBS_ERR_MISALIGNED
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32_noalloc(ident, ok, ok, ok, ok, None)
    assert e.value.status == B.CBS_ERR_UNSUPPORTED


def test_two_input_plans(cuda_lib):
    """Channel-concatenation layers: what each variant accepts, the per-input
    byte counts, and the entry points that refuse them (no launch)."""
    ok = 1 << 20
    # CUDA-core FP32, both layouts: x holds c_in - c_in_b channels, x_b the rest
    for lay in (B.CBS_NCHW, B.CBS_NHWC):
        p = B.cbs_plan(make_desc(2, 384, 40, 40, 128, 1, 1, in_layout=lay, c_in_b=128,
                                 force_variant=B.CBS_VARIANT_SIMT_FP32))
        assert p.variant == B.CBS_VARIANT_SIMT_FP32
        assert p.x_bytes == 2 * 40 * 40 * 256 * 4 and p.x_b_bytes == 2 * 40 * 40 * 128 * 4
    # tensor cores: a channel block never straddles the two inputs
    for prec, eb in ((B.CBS_BF16, 2), (B.CBS_TF32, 4)):
        p = B.cbs_plan(make_desc(2, 384, 40, 40, 128, 1, 1, prec=prec, c_in_b=128))
        assert (256 * eb) % (p.block_k * eb) == 0
        assert p.x_bytes == 2 * 40 * 40 * 256 * eb and p.x_b_bytes == 2 * 40 * 40 * 128 * eb
        p = B.cbs_plan(make_desc(1, 48, 20, 20, 64, 3, 1, prec=prec, c_in_b=16))
        assert (32 % p.block_k) == 0 and p.x_b_bytes == 20 * 20 * (p.c_in_pad - 32) * eb
    assert B.cbs_plan(make_desc(1, 24, 20, 20, 64, 3, 1, prec=B.CBS_BF16, c_in_b=8)).c_in_pad == 32
    # INT8: channel blocks of 64/32/16 codes that also divide the first input
    p8 = B.cbs_plan(make_desc(2, 96, 20, 20, 64, 3, 1, prec=B.CBS_INT8, c_in_b=32))
    assert p8.variant == B.CBS_VARIANT_TC_INT8 and 64 % p8.block_k == 0 and p8.block_k == 32
    assert p8.x_bytes == 2 * 400 * 64 and p8.x_b_bytes == 2 * 400 * 32
    rejects = [
        (dict(c_in=16, c_in_b=16), B.CBS_ERR_INVALID_ARG),                      # c_in_b must be < c_in
        (dict(c_in=16, c_in_b=-1), B.CBS_ERR_INVALID_ARG),
        (dict(c_in=40, c_in_b=16, prec=B.CBS_INT8), B.CBS_ERR_UNSUPPORTED),     # first input 24 codes: not 16-aligned
        (dict(c_in=24, c_in_b=16, prec=B.CBS_BF16), B.CBS_ERR_UNSUPPORTED),     # first input 8 bf16 = 16 B
        (dict(c_in=36, c_in_b=4, prec=B.CBS_BF16), B.CBS_ERR_UNSUPPORTED),      # second input 4 bf16 = 8 B
        (dict(c_in=4, c_in_b=2, force_variant=B.CBS_VARIANT_STEM), B.CBS_ERR_UNSUPPORTED),
    ]
    for kw, status in rejects:
        prec = kw.pop("prec", B.CBS_FP32)
        c_in = kw.pop("c_in")
        lay = B.CBS_NHWC if prec != B.CBS_FP32 else B.CBS_NCHW
        with pytest.raises(B.CbsError) as e:
            B.cbs_plan(make_desc(1, c_in, 20, 20, 32, 3, 1, prec=prec, in_layout=lay, **kw))
        assert e.value.status == status, (c_in, kw)
    # a small-channel two-input layer takes the implicit GEMM, not the stem
    assert B.cbs_plan(make_desc(1, 4, 20, 20, 16, 3, 1, c_in_b=2)).variant == B.CBS_VARIANT_SIMT_FP32
    two = B.cbs_plan(make_desc(1, 64, 20, 20, 32, 3, 1, c_in_b=32))
    one = B.cbs_plan(make_desc(1, 64, 20, 20, 32, 3, 1))
    ws = two.workspace_bytes
    for call in (lambda: B.cbs_conv_bn_silu_f32(two, ok, ok, ok, ok, ok, ws, None),
                 lambda: B.cbs_conv_bn_act(two, ok, ok, ok, None, ok, ok, ws, None),
                 lambda: B.cbs_conv_bn_act_cat(one, ok, ok, ok, ok, None, ok, ok, one.workspace_bytes, None),
                 lambda: B.cbs_conv_bn_act_cat(two, ok, None, ok, ok, None, ok, ok, ws, None)):
        with pytest.raises(B.CbsError) as e:
            call()
        assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_act_cat(two, ok, ok + 8, ok, ok, None, ok, ok, ws, None)
    assert e.value.status == B.CBS_ERR_MISALIGNED
    for call, status in ((lambda: B.cbs_pack_input(two, ok, ok, 0.0, None), B.CBS_ERR_UNSUPPORTED),
                         (lambda: B.cbs_conv_bn_silu_f32_noalloc(two, ok, ok, ok, ok, None), B.CBS_ERR_UNSUPPORTED)):
        with pytest.raises(B.CbsError) as e:
            call()
        assert e.value.status == status


def test_launch_options(cuda_lib):
    """Programmatic dependent launch is on by default and can be switched."""
    assert B.cbs_launch_options() == B.CBS_LAUNCH_PDL
    try:
        B.cbs_set_launch_options(0)
        assert B.cbs_launch_options() == 0
        with pytest.raises(B.CbsError) as e:
            B.cbs_set_launch_options(6)
        assert e.value.status == B.CBS_ERR_INVALID_ARG
        assert B.cbs_launch_options() == 0
    finally:
        B.cbs_set_launch_options(B.CBS_LAUNCH_PDL)


def test_zero_point_plans(cuda_lib):
    """INT8 zero points: range checks, INT8 only; the plan's buffers do not
    change."""
    sym = B.cbs_plan(make_desc(2, 32, 20, 20, 48, 3, 1, prec=B.CBS_INT8))
    asym = B.cbs_plan(make_desc(2, 32, 20, 20, 48, 3, 1, prec=B.CBS_INT8, zero_point_x=-7, zero_point_y=100))
    assert asym.w_packed_bytes == sym.w_packed_bytes == 48 * sym.k_gemm * 2
    assert (asym.block_n, asym.stages, asym.k_group) == (sym.block_n, sym.stages, sym.k_group)
    stem = B.cbs_plan(make_desc(1, 3, 64, 64, 16, 3, 2, prec=B.CBS_INT8, zero_point_x=12))
    assert stem.variant == B.CBS_VARIANT_STEM
    for kw, prec in ((dict(zero_point_x=128), B.CBS_INT8), (dict(zero_point_y=-129), B.CBS_INT8),
                     (dict(zero_point_x=1), B.CBS_BF16), (dict(zero_point_y=1), B.CBS_FP32)):
        lay = B.CBS_NCHW if prec == B.CBS_FP32 else B.CBS_NHWC
        with pytest.raises(B.CbsError) as e:
            B.cbs_plan(make_desc(1, 32, 20, 20, 48, 3, 1, prec=prec, in_layout=lay, **kw))
        assert e.value.status == B.CBS_ERR_INVALID_ARG


def test_maxpool_argument_rules(cuda_lib):
    ok = 1 << 20
    for args in ((1, 8, 10, 10, 3, 1, 2), (1, 8, 10, 10, 0, 1, 0), (1, 8, 2, 2, 5, 1, 1), (1, 0, 10, 10, 3, 1, 1),
                 (1, 8, 10, 10, 3, 0, 1)):
        with pytest.raises(B.CbsError) as e:
            B.cbs_maxpool2d(ok, ok, *args, B.CBS_NHWC, B.CBS_FP32, None)
        assert e.value.status == B.CBS_ERR_INVALID_ARG, args
    with pytest.raises(B.CbsError) as e:
        B.cbs_maxpool2d(ok, ok, 1, 8, 10, 10, 5, 1, 2, 7, B.CBS_FP32, None)
    assert e.value.status == B.CBS_ERR_INVALID_ARG
    with pytest.raises(B.CbsError) as e:
        B.cbs_maxpool2d(ok + 4, ok, 1, 8, 10, 10, 5, 1, 2, B.CBS_NHWC, B.CBS_FP32, None)
    assert e.value.status == B.CBS_ERR_MISALIGNED
    B.cbs_maxpool2d(ok, ok, 0, 8, 10, 10, 5, 1, 2, B.CBS_NHWC, B.CBS_FP32, None)   # empty batch: nothing enqueued


def test_split_k_plan_rules(cuda_lib):
    """Tensor-core split-K on request (the cost model keeps one part); it
    needs im2col A and streamed weights."""
    auto = B.cbs_plan(make_desc(16, 128, 40, 40, 128, 3, 1, prec=B.CBS_BF16, force_block_m=256, force_block_n=128))
    assert auto.split_k == 1 and auto.workspace_bytes == 0
    forced = B.cbs_plan(make_desc(16, 128, 40, 40, 128, 3, 1, prec=B.CBS_BF16, force_block_m=256, force_block_n=128,
                                  force_split_k=3))
    assert forced.split_k == 3 and forced.grid_ctas == 152
    assert forced.workspace_bytes == 3328 + 100 * 3 * 256 * 128 * 4   # counters [tile][8 warps], then partials
    for kw in ({"force_window": 1}, {"force_b_resident": 1}):
        with pytest.raises(B.CbsError) as e:
            B.cbs_plan(make_desc(2, 64, 16, 16, 64, 3, 1, prec=B.CBS_BF16, force_split_k=2, **kw))
        assert e.value.status == B.CBS_ERR_UNSUPPORTED


@pytest.mark.parametrize("prec,n", [(B.CBS_BF16, 16), (B.CBS_INT8, 16), (B.CBS_FP32, 1)])
def test_plan_follows_the_sm_count(cuda_lib, prec, n):
    """num_sms = 0 plans for the GB300's 152 SMs; another count sizes the
    persistent grids (at most one CTA per SM for the tensor-core kernels)
    and the waves for that device."""
    layout = B.CBS_NHWC if prec != B.CBS_FP32 else B.CBS_NCHW
    for i, s in enumerate(wl.LAYER_LIST[1:], start=1):
        d0 = make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, prec=prec, in_layout=layout, num_sms=0)
        d152 = make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, prec=prec, in_layout=layout, num_sms=152)
        d76 = make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, prec=prec, in_layout=layout, num_sms=76)
        p0, p152, p76 = B.cbs_plan(d0), B.cbs_plan(d152), B.cbs_plan(d76)
        assert bytes(p0)[:ctypes.sizeof(B.cbs_plan_t) - ctypes.sizeof(B.cbs_layer_desc)] == \
            bytes(p152)[:ctypes.sizeof(B.cbs_plan_t) - ctypes.sizeof(B.cbs_layer_desc)], i
        if p76.variant in (B.CBS_VARIANT_TC_TF32, B.CBS_VARIANT_TC_BF16, B.CBS_VARIANT_TC_INT8,
                           B.CBS_VARIANT_TC_TF32X3):
            assert p76.grid_ctas <= 76 and p152.grid_ctas <= 152, i
            assert p152.grid_ctas == min(152, p152.m_tiles * p152.n_tiles * p152.split_k) or p152.b_resident, i
    with pytest.raises(B.CbsError) as e:
        B.cbs_plan(make_desc(1, 16, 40, 40, 32, 3, 1, num_sms=-1))
    assert e.value.status == B.CBS_ERR_INVALID_ARG


def _ksteps(plan):
    """K steps of a TF32/BF16 plan: block_k channels per step, every tap."""
    return plan.desc.k * plan.desc.k * (plan.c_in_pad // plan.block_k)


@pytest.mark.parametrize("prec", [B.CBS_BF16, B.CBS_TF32])
def test_issuer_split_plan_invariants(cuda_lib, prec):
    """Every plan that splits a tile's K stages between the two MMA issuers
    has 128-pixel tiles, im2col A, one K part, an even pipeline depth (each
    ring slot then always feeds the same issuer), two or more stages per tile
    and an N tile of at most 128 (two accumulators per TMEM buffer)."""
    shapes = list(wl.LAYER_LIST[1:]) + [cl.spec for cl in wl.chain_layers(sppf=True)]
    seen = 0
    for s in shapes:
        for n in (1, 16):
            for kw in ({}, {"force_issuer_split": 1}, {"force_block_m": 128}, {"force_k_group": 3}):
                try:
                    pl = B.cbs_plan(make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, prec=prec, **kw))
                except B.CbsError as e:
                    assert e.status == B.CBS_ERR_UNSUPPORTED and kw, (s, kw)
                    continue
                if pl.variant == B.CBS_VARIANT_STEM:
                    assert pl.issuer_split == 1
                    continue
                assert pl.issuer_split in (1, 2)
                if kw.get("force_issuer_split") == 1:
                    assert pl.issuer_split == 2, (s, n)
                else:
                    assert pl.issuer_split == 1, (s, n, kw)     # on request only
                if pl.issuer_split == 2:
                    seen += 1
                    assert pl.block_m == 128 and pl.window == 0 and pl.split_k == 1, (s, n, kw)
                    assert pl.stages % 2 == 0 and pl.stages >= 2, (s, n, kw)
                    assert _ksteps(pl) // pl.k_group >= 2 and pl.block_n <= 128, (s, n, kw)
    assert seen > 0


def test_issuer_split_plan_rules(cuda_lib):
    """force_issuer_split: 0 and -1 keep one issuer per 128-pixel tile; 1
    where no configuration can take it, or on another variant, is refused;
    other values are invalid."""
    d = dict(n=16, c_in=64, h=40, w=40, c_out=128, k=3, stride=1, prec=B.CBS_BF16)
    for v in (0, -1):
        assert B.cbs_plan(make_desc(force_issuer_split=v, **d)).issuer_split == 1
    forced = B.cbs_plan(make_desc(force_issuer_split=1, **d))
    assert forced.issuer_split == 2 and forced.block_m == 128 and forced.stages % 2 == 0
    refused = [
        dict(d, force_block_m=256),                                  # 256-pixel tiles have two sub-tile issuers
        dict(d, force_window=1),                                     # windowed A
        dict(d, force_split_k=2),                                    # split-K
        dict(d, c_in=32, k=1, force_k_group=1, prec=B.CBS_BF16),     # one K step: one stage per tile
        dict(d, c_out=256, force_block_n=256),                       # N tile over 128
        dict(d, prec=B.CBS_INT8),                                    # another variant
        dict(n=1, c_in=64, h=40, w=40, c_out=128, k=3, stride=1, prec=B.CBS_FP32),
    ]
    for kw in refused:
        with pytest.raises(B.CbsError) as e:
            B.cbs_plan(make_desc(force_issuer_split=1, **kw))
        assert e.value.status == B.CBS_ERR_UNSUPPORTED, kw
    for v in (2, -2):
        with pytest.raises(B.CbsError) as e:
            B.cbs_plan(make_desc(force_issuer_split=v, **d))
        assert e.value.status == B.CBS_ERR_INVALID_ARG
