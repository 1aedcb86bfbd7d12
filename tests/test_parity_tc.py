"""GPU parity of the tcgen05 tensor-core paths (TF32, BF16) against the CPU
FP32 oracle.

Bars: relative L2 <= 5e-3 over the whole output against the oracle on the
float32 input the library receives (this covers the whole path: TF32
operands truncated by the tensor cores, BF16 inputs and weights rounded to
bfloat16, FP32 accumulation, bfloat16 output); and max |err| / max(1, |ref|)
<= 2e-2.  TF32 takes the max bound against the same oracle.  For BF16 the
max bound is taken against the oracle on the bfloat16 operands the layer
multiplies (x and the folded weights rounded to nearest even): an
exact-arithmetic layer on bfloat16 operands already exceeds 2e-2 against
the float32 input (tests/test_parity_bar.py)."""
import numpy as np
import pytest
import torch

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import check_tc, nhwc_to_nchw, tc_refs

pytestmark = pytest.mark.gpu

PRECS = {"tf32": B.CBS_TF32, "bf16": B.CBS_BF16}


def run_tc(spec, x, p, prec, out_layout=B.CBS_NHWC, **kw):
    n = x.shape[0]
    desc = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                     prec=prec, in_layout=B.CBS_NHWC, out_layout=out_layout, **kw)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xp = layer.pack_input(torch.from_numpy(x).cuda())
    y = layer(xp)
    torch.cuda.synchronize()
    y = y.float().cpu().numpy()
    if out_layout == B.CBS_NHWC:
        y = nhwc_to_nchw(y)
    return y, layer


def check(y, spec, x, p, prec, what=""):
    check_tc(prec, y, tc_refs(prec, x, p, spec.stride, spec.pad), what)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
def test_tiny_first(cuda_lib, prec):
    """Smallest case: one 128-pixel tile, one K step per tap."""
    spec = wl.LayerSpec(16, 16, 3, 1, 8)
    x, p = wl.layer_inputs(spec, 2, layer_index=2)
    y, _ = run_tc(spec, x, p, PRECS[prec])
    check(y, spec, x, p, prec)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
def test_single_layer_40x40(cuda_lib, prec):
    spec = wl.SINGLE_LAYER
    x, p = wl.layer_inputs(spec, 1)
    for out_layout in (B.CBS_NHWC, B.CBS_NCHW):
        y, _ = run_tc(spec, x, p, PRECS[prec], out_layout=out_layout)
        check(y, spec, x, p, prec, out_layout)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("i", range(len(wl.LAYER_LIST)))
def test_layer_list_batch1(cuda_lib, prec, i):
    spec = wl.LAYER_LIST[i]
    x, p = wl.layer_inputs(spec, 1, layer_index=i)
    y, layer = run_tc(spec, x, p, PRECS[prec])
    check(y, spec, x, p, prec, (i, layer.plan.block_n, layer.plan.block_k, layer.plan.stages))


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("shape", [
    (3, 16, 48, 3, 2, 13),     # ragged pixels, stride 2, BN = 48
    (2, 32, 16, 1, 1, 11),     # 1x1, tail tile
    (1, 64, 272, 3, 1, 6),     # C_out > 256: two N tiles, second ragged
    (4, 48, 32, 3, 1, 9),      # C_in = 48 (96 B in BF16: 32-byte K steps)
    (1, 3, 16, 3, 2, 34),      # C_in = 3 padded, stride 2, even size
    (2, 8, 16, 3, 1, 1),       # 1x1 image with a 3x3 filter
    (1, 4, 64, 7, 2, 21),      # direct small-channel kernel, 7x7: 49 KB of weights
    (2, 16, 20, 3, 1, 9),      # BF16 rows of 40 bytes: direct stores; TF32 rows of 80: staged stores
    (1, 32, 36, 1, 1, 7),      # C_out = 36: ragged channel block in both store paths
])
def test_ragged(cuda_lib, prec, shape):
    n, c_in, c_out, k, stride, h = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=9)
    y, _ = run_tc(spec, x, p, PRECS[prec])
    check(y, spec, x, p, prec, shape)


@pytest.mark.parametrize("out_layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("shape", [
    (2, 3, 16, 3, 2, 38, 38),      # 3x3 s2 with an even width: pixel-pair copies, ragged last tile
    (2, 3, 16, 3, 2, 37, 37),      # odd width: one copy per tap
    (1, 4, 32, 3, 1, 19, 19),      # stride 1
    (3, 1, 48, 1, 1, 9, 9),        # 1x1 filter: one K slice, C_out 48
    (1, 2, 64, 3, 2, 50, 34),      # C_out 64, non-square
    (1, 3, 40, 3, 2, 30, 30),      # C_out 40: a ragged 16-channel block
    (1, 3, 20, 3, 2, 22, 22),      # C_out 20: per-channel stores
    (8, 3, 16, 3, 2, 256, 256),    # 1024 tiles: several per persistent CTA, through the whole ring
])
def test_tensor_core_stem(cuda_lib, out_layout, shape):
    """BF16 layers with at most 4 input channels and k <= 3 run on the
    tensor-core stem kernel."""
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=4)
    y, layer = run_tc(spec, x, p, B.CBS_BF16, out_layout=out_layout)
    pl = layer.plan
    assert pl.variant == B.CBS_VARIANT_STEM and pl.block_m == 128
    sms = layer.desc.num_sms
    if pair_stem_kernel(spec, out_layout):
        assert pl.threads == 288 and pl.grid_ctas == min(n * spec.oh, sms * 2)   # bands of output rows, two CTAs per SM
    else:
        assert pl.threads == 256
        assert pl.grid_ctas == min(pl.m_tiles, sms * (5 if c_out <= 32 else 4))   # 4 x 128 TMEM columns for wide C_out
    check(y, spec, x, p, "bf16", shape)


def pair_stem_kernel(spec, out_layout):
    """The shapes the stem's row kernel takes: 3x3, stride 2, pad 1, even
    input width up to 1024, 16 output channels, NHWC output."""
    return (spec.k == 3 and spec.stride == 2 and spec.pad == 1 and spec.width % 2 == 0 and spec.c_out == 16
            and out_layout == B.CBS_NHWC)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("act", [B.CBS_ACT_SILU, B.CBS_ACT_IDENTITY])
@pytest.mark.parametrize("shape", [
    (1, 3, 16, 3, 2, 2, 2),        # one output pixel: one pair of tiles, the second empty
    (3, 3, 16, 3, 2, 37, 38),      # odd height: the last output row's third kernel row is padding
    (2, 4, 16, 3, 2, 30, 62),      # four channels, non-square, odd tile count
    (16, 3, 16, 3, 2, 320, 320),   # 2560 output rows: bands of ~8 rows, round the slot rings
    (2, 3, 16, 3, 2, 640, 640),    # the detector's width: three M tiles per output row, the last ragged
    (5, 3, 16, 3, 2, 9, 200),      # bands that cross images (output row 0 inside a band)
])
def test_stem_pair_kernel(cuda_lib, prec, act, shape):
    """The BF16 and TF32 stems' row kernel (TMA input rows, rewritten in
    shared memory as MMA operand rows) against the oracle, with and without
    SiLU."""
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    assert pair_stem_kernel(spec, B.CBS_NHWC)
    x, p = wl.layer_inputs(spec, n, layer_index=4)
    y, layer = run_tc(spec, x, p, PRECS[prec], activation=act)
    assert layer.plan.variant == B.CBS_VARIANT_STEM and layer.plan.threads == 288
    ctas = 2 if prec == "bf16" else 1   # the TF32 rows take twice the shared memory
    assert layer.plan.grid_ctas == min(n * spec.oh, layer.desc.num_sms * ctas)
    check_tc(prec, y, tc_refs(prec, x, p, spec.stride, spec.pad, act=act), (shape, act))


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
def test_non_square_image(cuda_lib, prec):
    """H != W pins the order of the im2col corner and offset coordinates."""
    spec = wl.LayerSpec(32, 32, 3, 1, 12, 20)
    x, p = wl.layer_inputs(spec, 2, layer_index=3)
    y, _ = run_tc(spec, x, p, PRECS[prec])
    check(y, spec, x, p, prec)
    spec2 = wl.LayerSpec(32, 64, 3, 2, 18, 10)
    x2, p2 = wl.layer_inputs(spec2, 1, layer_index=4)
    y2, _ = run_tc(spec2, x2, p2, PRECS[prec])
    check(y2, spec2, x2, p2, prec)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("bn", [16, 32, 64, 128, 256])
def test_forced_block_n(cuda_lib, prec, bn):
    spec = wl.LayerSpec(64, 256, 3, 1, 10)
    x, p = wl.layer_inputs(spec, 2, layer_index=8)
    y, layer = run_tc(spec, x, p, PRECS[prec], force_block_n=bn)
    assert layer.plan.block_n == bn
    check(y, spec, x, p, prec, bn)


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("i", range(len(wl.LAYER_LIST)))
def test_batch16_layer_list(cuda_lib, prec, i):
    """The batch-16 config: every list layer, every one of the 16 images
    against the oracle (tiles run over flattened (n, oh, ow), so most tiles
    of the middle images cross an image boundary)."""
    spec = wl.LAYER_LIST[i]
    x, p = wl.layer_inputs(spec, 16, layer_index=i)
    y, layer = run_tc(spec, x, p, PRECS[prec])
    assert y.shape[0] == 16 and np.isfinite(y).all()
    check(y, spec, x, p, prec, (i, layer.plan.block_m, layer.plan.block_n))


CONFIGS = [(prec, bm, kg, bres) for prec in ("bf16", "tf32")
           for bm, kg, bres in ((128, 1, -1), (128, 3, 1), (256, 1, 1), (256, 3, -1), (256, 3, 1), (128, 1, 1))]
CONFIGS.append(("bf16", 128, 9, -1))   # a whole 3x3 window per stage


@pytest.mark.parametrize("prec,bm,kg,bres", CONFIGS)
@pytest.mark.parametrize("shape", [
    (2, 32, 64, 3, 1, 20, 64),     # several 256-pixel tiles with a ragged tail
    (3, 32, 48, 3, 2, 17, 48),     # stride 2, BN = 48 (B tiles not a multiple of 1 KB)
    (2, 32, 272, 3, 1, 9, 96),     # several N tiles, the last ragged: resident weights pin one N tile per CTA
])
def test_tile_height_k_group_resident_weights(cuda_lib, prec, bm, kg, bres, shape):
    """Every combination of tile height (one or two 128-pixel sub-tiles per
    TMA box), K steps per pipeline stage and resident or streamed weights.
    The N tile is forced where shared memory holds it, else chosen."""
    n, c_in, c_out, k, stride, h, bn = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=11)
    kw = dict(force_block_m=bm, force_k_group=kg, force_b_resident=bres)
    try:
        B.cbs_plan(make_desc(n, c_in, h, h, c_out, k, stride, prec=PRECS[prec], force_block_n=bn, **kw))
        kw["force_block_n"] = bn
    except B.CbsError as e:
        assert e.status == B.CBS_ERR_UNSUPPORTED
    y, layer = run_tc(spec, x, p, PRECS[prec], **kw)
    pl = layer.plan
    assert (pl.block_m, pl.k_group, pl.b_resident) == (bm, kg, 1 if bres > 0 else 0)
    check(y, spec, x, p, prec, (shape, bm, kg, bres, pl.block_n, pl.stages))


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("bm,bres", [(128, -1), (128, 1), (256, -1), (256, 1)])
def test_pointwise_tall_tiles(cuda_lib, prec, bm, bres):
    """1x1 layer (A loaded as a 2-D tile of 128 or 256 rows), ragged pixel count."""
    spec = wl.LayerSpec(64, 96, 1, 1, 13)
    x, p = wl.layer_inputs(spec, 4, layer_index=12)
    y, layer = run_tc(spec, x, p, PRECS[prec], force_block_m=bm, force_b_resident=bres, force_k_group=1)
    assert (layer.plan.block_m, layer.plan.b_resident) == (bm, 1 if bres > 0 else 0)
    check(y, spec, x, p, prec, (bm, bres))



WINDOW_SHAPES = [  # (n, c_in, c_out, k, h, w, N tile tried first)
    (2, 64, 64, 3, 20, 20, 64),      # several tiles per image, last one ragged
    (1, 128, 96, 3, 13, 17, 96),     # non-square, window rows of 19 positions
    (1, 64, 32, 5, 11, 11, 32),      # 5x5 filter, pad 2
    (3, 64, 48, 1, 9, 9, 48),        # 1x1 through the window path
    (1, 192, 272, 3, 7, 7, 128),     # three channel blocks (BF16), several N tiles, the last ragged
]


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("bm,bres", [(128, -1), (256, -1), (128, 1), (256, 1)])
@pytest.mark.parametrize("shape", WINDOW_SHAPES)
def test_windowed_a(cuda_lib, prec, bm, bres, shape):
    """Stride-1 layers with the windowed A operand: one zero-padded input
    window per tile and channel block, every tap a shifted view of it, weights
    resident or streamed through the weight ring.  Resident weights that do
    not fit fall back to the ring."""
    n, c_in, c_out, k, h, w, bn = shape
    spec = wl.LayerSpec(c_in, c_out, k, 1, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=13)
    kw = None
    for cand in (dict(force_block_n=bn, force_b_resident=bres), dict(force_b_resident=bres),
                 dict(force_block_n=bn, force_b_resident=-1), dict(force_b_resident=-1)):
        cand.update(force_window=1, force_block_m=bm)
        try:
            B.cbs_plan(make_desc(n, c_in, h, w, c_out, k, 1, prec=PRECS[prec], **cand))
            kw = cand
            break
        except B.CbsError as e:
            assert e.status == B.CBS_ERR_UNSUPPORTED
    assert kw is not None
    y, layer = run_tc(spec, x, p, PRECS[prec], **kw)
    pl = layer.plan
    assert pl.window == 1 and pl.block_m == bm
    check(y, spec, x, p, prec, (shape, bm, pl.b_resident, pl.block_n, pl.stages, pl.k_group))


ISSUER_SPLIT_SHAPES = [  # (n, c_in, c_out, k, stride, h, K steps per stage, resident weights)
    (2, 32, 64, 3, 1, 20, 3, -1),     # 3 stages per tile (odd): a tile's first stage alternates issuers
    (2, 32, 64, 3, 1, 20, 3, 1),      # the same with resident weights
    (8, 32, 64, 3, 1, 80, 3, -1),     # 400 tiles: up to three per CTA, both TMEM buffers reused
    (3, 32, 48, 3, 2, 17, 1, -1),     # 9 stages, stride 2, N tile 48, ragged pixels
    (2, 32, 200, 3, 1, 9, 1, 1),      # two N tiles, the second ragged; resident weights
    (4, 128, 96, 1, 1, 13, 1, -1),    # 1x1, ragged pixel count
    (1, 64, 40, 3, 2, 17, 1, -1),     # ragged output channels
]


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("shape", ISSUER_SPLIT_SHAPES)
def test_issuer_split(cuda_lib, prec, shape):
    """128-pixel tiles whose K stages alternate between the two MMA issuers
    (each into its own accumulator, added by the epilogue; on request)
    against the oracle, beside the same plan with one issuer; repeated calls
    agree."""
    n, c_in, c_out, k, stride, h, kg, bres = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=19)
    kw = dict(force_block_m=128, force_k_group=kg, force_b_resident=bres)
    y, layer = run_tc(spec, x, p, PRECS[prec], force_issuer_split=1, **kw)
    pl = layer.plan
    ksteps = k * k * (pl.c_in_pad // pl.block_k)
    assert pl.issuer_split == 2 and pl.block_m == 128 and pl.stages % 2 == 0, (pl.issuer_split, pl.stages)
    assert (pl.k_group, pl.b_resident) == (kg, 1 if bres > 0 else 0)
    if shape[:6] == (2, 32, 64, 3, 1, 20):
        assert (ksteps // kg) % 2 == 1     # the odd stage count is what the case is for
    check(y, spec, x, p, prec, (shape, pl.block_n, pl.stages, ksteps // kg))
    y_again, _ = run_tc(spec, x, p, PRECS[prec], force_issuer_split=1, **kw)
    assert np.array_equal(y, y_again)
    y_one, one = run_tc(spec, x, p, PRECS[prec], force_issuer_split=-1, **kw)
    assert one.plan.issuer_split == 1
    check(y_one, spec, x, p, prec, (shape, "one issuer"))


def test_issuer_split_with_residual_two_inputs_and_identity(cuda_lib):
    """The issuer split beside the residual add, the channel concatenation
    and the identity activation."""
    spec = wl.LayerSpec(96, 64, 3, 1, 14)
    x, p = wl.layer_inputs(spec, 2, layer_index=20)
    r = np.random.default_rng(5).standard_normal((2, 64, 14, 14)).astype(np.float32)
    for act in (B.CBS_ACT_SILU, B.CBS_ACT_IDENTITY):
        desc = make_desc(2, 96, 14, 14, 64, 3, 1, prec=B.CBS_BF16, force_issuer_split=1, residual=1, c_in_b=32,
                         activation=act)
        layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
        assert layer.plan.issuer_split == 2
        xa, xb = layer.pack_inputs(torch.from_numpy(np.ascontiguousarray(x[:, :64])).cuda(),
                                   torch.from_numpy(np.ascontiguousarray(x[:, 64:])).cuda())
        rr = torch.from_numpy(np.ascontiguousarray(r.transpose(0, 2, 3, 1))).cuda().to(torch.bfloat16)
        y = nhwc_to_nchw(layer(xa, residual=rr, x_b=xb).float().cpu().numpy())
        rb = torch.from_numpy(r).to(torch.bfloat16).float().numpy()
        check_tc("bf16", y, tc_refs("bf16", x, p, 1, 1, act=act, residual=rb), act)


WINDOW_S2_SHAPES = [  # (n, c_in, c_out, h, w, N tile tried first): 3x3, stride 2, pad 1
    (2, 16, 32, 64, 64, 32),         # 32-byte pixels (BF16), several tiles per image
    (2, 32, 64, 40, 40, 64),         # 64-byte pixels (BF16), 64-byte TF32 pixels with 16 channels below
    (1, 16, 48, 17, 18, 48),         # odd height: the planes have 9 and 8 rows; ragged last tile
    (3, 8, 40, 9, 14, 48),           # 8 channels (TF32: 32-byte pixels), ragged output channels
    (1, 16, 200, 12, 12, 128),       # several N tiles, the last ragged
    (2, 16, 16, 2, 2, 16),           # one output pixel per image: every tap but one in the padding
]


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("bm,bres", [(128, -1), (256, -1), (128, 1), (256, 1)])
@pytest.mark.parametrize("shape", WINDOW_S2_SHAPES)
def test_windowed_a_stride2(cuda_lib, prec, bm, bres, shape):
    """3x3 stride-2 layers with the windowed A operand: per tile, one box of
    the even input rows and one of the odd rows, each row read as pairs of
    pixels; every tap a view of one of them.  Resident weights that do not
    fit fall back to the weight ring; shapes whose window does not fit
    shared memory are refused by the planner."""
    n, c_in, c_out, h, w, bn = shape
    spec = wl.LayerSpec(c_in, c_out, 3, 2, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=21)
    kw = None
    for cand in (dict(force_block_n=bn, force_b_resident=bres), dict(force_b_resident=bres),
                 dict(force_block_n=bn, force_b_resident=-1), dict(force_b_resident=-1)):
        cand.update(force_window=1, force_block_m=bm)
        try:
            B.cbs_plan(make_desc(n, c_in, h, w, c_out, 3, 2, prec=PRECS[prec], **cand))
            kw = cand
            break
        except B.CbsError as e:
            assert e.status == B.CBS_ERR_UNSUPPORTED
    if kw is None:
        pytest.skip("window does not fit shared memory")
    for out_layout in (B.CBS_NHWC, B.CBS_NCHW):
        y, layer = run_tc(spec, x, p, PRECS[prec], out_layout=out_layout, **kw)
        pl = layer.plan
        assert pl.window == 1 and pl.block_m == bm
        check(y, spec, x, p, prec, (shape, bm, pl.b_resident, pl.block_n, pl.stages, pl.k_group, out_layout))
    y2, _ = run_tc(spec, x, p, PRECS[prec], out_layout=B.CBS_NCHW, **kw)
    assert np.array_equal(y, y2)


def test_no_timeout_reported(cuda_lib):
    assert B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream) == B.CBS_OK


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("case", [
    ((2, 64, 64, 3, 1, 20), 2, {}),                        # two K parts
    ((2, 64, 64, 3, 1, 20), 3, {"force_block_m": 256}),    # tall tiles: each warp owns a whole sub-tile
    ((1, 64, 40, 3, 2, 17), 5, {"force_k_group": 1}),      # ragged pixels and channels; 5 parts over 9 stages
    ((2, 128, 96, 1, 1, 9), 2, {"force_block_n": 48}),     # 1x1, several N tiles
])
def test_split_k(cuda_lib, prec, case):
    """K split over parts whose partial tiles the last-arriving epilogue warp
    of each region sums in order (NHWC and NCHW outputs)."""
    (n, c_in, c_out, k, stride, h), split, kw = case
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=17)
    for out_layout in (B.CBS_NHWC, B.CBS_NCHW):
        y, layer = run_tc(spec, x, p, PRECS[prec], out_layout=out_layout, force_split_k=split, **kw)
        assert layer.plan.split_k == split and layer.plan.workspace_bytes > 0
        check(y, spec, x, p, prec, (split, out_layout))
        y2, _ = run_tc(spec, x, p, PRECS[prec], out_layout=out_layout, force_split_k=split, **kw)
        assert np.array_equal(y, y2)     # the parts are summed in a fixed order


def test_split_k_with_residual_and_two_inputs(cuda_lib):
    """Split-K beside the residual add and the channel concatenation."""
    spec = wl.LayerSpec(96, 64, 3, 1, 14)
    x, p = wl.layer_inputs(spec, 2, layer_index=18)
    r = np.random.default_rng(4).standard_normal((2, 64, 14, 14)).astype(np.float32)
    desc = make_desc(2, 96, 14, 14, 64, 3, 1, prec=B.CBS_BF16, force_split_k=3, residual=1, c_in_b=32)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    assert layer.plan.split_k == 3
    xa, xb = layer.pack_inputs(torch.from_numpy(np.ascontiguousarray(x[:, :64])).cuda(),
                               torch.from_numpy(np.ascontiguousarray(x[:, 64:])).cuda())
    rr = torch.from_numpy(np.ascontiguousarray(r.transpose(0, 2, 3, 1))).cuda().to(torch.bfloat16)
    y = nhwc_to_nchw(layer(xa, residual=rr, x_b=xb).float().cpu().numpy())
    r = torch.from_numpy(r).to(torch.bfloat16).float().numpy()
    check_tc("bf16", y, tc_refs("bf16", x, p, 1, 1, residual=r))
    for _ in range(3):   # the arrival counters are back at zero after every call
        again = nhwc_to_nchw(layer(xa, residual=rr, x_b=xb).float().cpu().numpy())
        assert np.array_equal(again, y)



@pytest.mark.parametrize("out_layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("shape", [
    (2, 3, 16, 3, 2, 38, 38),      # the stem's shape, ragged last tile
    (2, 3, 16, 3, 2, 37, 37),      # odd width
    (1, 4, 32, 3, 1, 19, 19),      # stride 1
    (3, 1, 48, 1, 1, 9, 9),        # 1x1: one K slice
    (1, 2, 64, 2, 2, 50, 34),      # 2x2 filter (4 taps), C_out 64
    (1, 3, 20, 3, 2, 22, 22),      # C_out 20: per-channel stores
    (4, 3, 16, 3, 2, 160, 160),    # several tiles per persistent CTA
])
def test_tensor_core_stem_tf32(cuda_lib, out_layout, shape):
    """TF32 layers with at most 4 input channels and k <= 3 run on the TF32
    tensor-core stems (taps straight into 32-byte-swizzled K slices, or for
    the detector's 3x3 s2 16-channel NHWC case the row kernel)."""
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=5)
    y, layer = run_tc(spec, x, p, B.CBS_TF32, out_layout=out_layout)
    pl = layer.plan
    assert pl.variant == B.CBS_VARIANT_STEM and pl.block_m == 128
    if pair_stem_kernel(spec, out_layout):
        assert pl.threads == 288 and pl.grid_ctas == min(n * spec.oh, layer.desc.num_sms)   # one CTA per SM
    else:
        assert pl.threads == 256 and pl.grid_ctas == min(pl.m_tiles, layer.desc.num_sms * 4)
    check(y, spec, x, p, "tf32", shape)
