"""GPU parity of the FP32 layer on the tensor cores (CBS_VARIANT_TC_TF32X3)
against the CPU oracle, at the FP32 bar (relative L2 <= 1e-5).

The variant splits every fp32 activation and weight into a TF32 head and the
remainder and sums three kind::tf32 products per K slice, so it must meet
the same bar as the CUDA-core FP32 kernel, which plain TF32 misses by about
two orders of magnitude (relative L2 ~1e-3).  Covered: 1x1 2-D tile loads
and im2col boxes, strides 1 and 2, ragged pixel tiles and channel counts
(C_in padded to 8, C_out not a multiple of 16), 32-, 64- and 128-byte
channel blocks, several K steps per stage, NCHW and NHWC output, the
identity activation with a residual, two inputs, and the plan and
workspace rules of the variant."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import TOL_FP32_REL_L2, nhwc_to_nchw, rel_l2

X3 = B.CBS_VARIANT_TC_TF32X3


def desc_x3(n, spec, out_layout=B.CBS_NHWC, **kw):
    return make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                     prec=B.CBS_FP32, in_layout=B.CBS_NHWC, out_layout=out_layout, force_variant=X3, **kw)


def run_x3(spec, x, p, out_layout=B.CBS_NHWC, **kw):
    layer = FusedConvBnSilu(desc_x3(x.shape[0], spec, out_layout, **kw), p.w, p.gamma, p.beta, p.mean, p.var,
                            p.eps)
    assert layer.plan.variant == X3
    y = layer(layer.pack_input(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    return (nhwc_to_nchw(y) if out_layout == B.CBS_NHWC else y), layer


def ref_of(spec, x, p):
    return oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad)


@pytest.mark.gpu
@pytest.mark.parametrize("out_layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("shape", [
    (2, 64, 64, 3, 1, 20, 20),       # im2col boxes, 128-byte channel blocks, 3x3 s1
    (1, 32, 96, 3, 2, 21, 19),       # stride 2, ragged pixel tile
    (2, 256, 128, 1, 1, 12, 12),     # 1x1: 2-D tile boxes, several K steps
    (1, 3, 16, 3, 2, 38, 38),        # C_in padded to 8: 32-byte channel blocks
    (1, 16, 20, 3, 1, 17, 13),       # 64-byte blocks, C_out 20 (ragged N tile)
    (1, 128, 256, 3, 2, 10, 10),     # wide N: several N tiles
])
def test_fp32_on_tensor_cores(cuda_lib, out_layout, shape):
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=31)
    y, _ = run_x3(spec, x, p, out_layout)
    e = rel_l2(y, ref_of(spec, x, p))
    assert e <= TOL_FP32_REL_L2, e


@pytest.mark.gpu
@pytest.mark.parametrize("c_in,kg", [(128, 1), (128, 2), (24, 3)])   # 48 KB or 12 KB per K step
def test_k_steps_per_stage(cuda_lib, c_in, kg):
    spec = wl.LayerSpec(c_in, 64, 3, 1, 14, 14)
    x, p = wl.layer_inputs(spec, 1, layer_index=32)
    y, layer = run_x3(spec, x, p, force_k_group=kg)
    assert layer.plan.k_group == kg
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.gpu
def test_list_layer_batch16_sample(cuda_lib):
    """A list layer at batch 16 (many tiles per persistent CTA): images 0 and
    15 against the oracle."""
    spec = wl.LAYER_LIST[5]
    x, p = wl.layer_inputs(spec, 16, layer_index=5)
    y, _ = run_x3(spec, x, p)
    for i in (0, 15):
        want = ref_of(spec, x[i:i + 1], p)
        assert rel_l2(y[i:i + 1], want) <= TOL_FP32_REL_L2


@pytest.mark.gpu
def test_identity_residual_and_two_inputs(cuda_lib):
    n, c_a, c_b, c_out, h = 1, 32, 32, 48, 11
    spec = wl.LayerSpec(c_a + c_b, c_out, 3, 1, h)
    x, p = wl.layer_inputs(spec, n, layer_index=33)
    r = np.random.default_rng(12).standard_normal((n, h, h, c_out)).astype(np.float32)
    desc = desc_x3(n, spec, activation=B.CBS_ACT_IDENTITY, residual=1, c_in_b=c_b)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xa, xb = layer.pack_inputs(torch.from_numpy(np.ascontiguousarray(x[:, :c_a])).cuda(),
                               torch.from_numpy(np.ascontiguousarray(x[:, c_a:])).cuda())
    y = layer(xa, residual=torch.from_numpy(r).cuda(), x_b=xb)
    torch.cuda.synchronize()
    want = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1, act=B.CBS_ACT_IDENTITY,
                                  residual=np.ascontiguousarray(r.transpose(0, 3, 1, 2)))
    assert rel_l2(nhwc_to_nchw(y.cpu().numpy()), want) <= TOL_FP32_REL_L2


@pytest.mark.gpu
def test_more_accurate_than_tf32(cuda_lib):
    """The split is what buys the accuracy: the same layer as plain TF32 is
    far off the FP32 bar."""
    spec = wl.LayerSpec(64, 64, 3, 1, 16, 16)
    x, p = wl.layer_inputs(spec, 1, layer_index=34)
    y3, _ = run_x3(spec, x, p)
    desc = make_desc(1, 64, 16, 16, 64, 3, 1, 1, prec=B.CBS_TF32, in_layout=B.CBS_NHWC, out_layout=B.CBS_NHWC)
    tf = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    yt = nhwc_to_nchw(tf(tf.pack_input(torch.from_numpy(x).cuda())).cpu().numpy())
    want = ref_of(spec, x, p)
    e3, et = rel_l2(y3, want), rel_l2(yt, want)
    assert e3 <= TOL_FP32_REL_L2 and et > 20 * e3, (e3, et)


def test_plan_rules(cuda_lib):
    """Host-side plan of the variant (no GPU call): FP32 only, NHWC input or
    NCHW (read by the kernel as given), both weight halves in w_packed,
    staged-kernel launch shape, split-K workspace."""
    spec = wl.LayerSpec(64, 96, 3, 1, 20, 20)
    pl = B.cbs_plan(desc_x3(2, spec))
    assert pl.variant == X3 and pl.block_m == 128 and pl.threads == 480
    assert pl.c_in_pad == 64 and pl.block_k == 32
    assert pl.w_packed_bytes == 2 * 96 * 9 * 64 * 4
    assert pl.x_bytes == 2 * 20 * 20 * 64 * 4
    # a layer with a wave of tiles or more runs unsplit; fewer tiles than SMs
    # take K parts to fill them
    big = B.cbs_plan(desc_x3(16, wl.LayerSpec(64, 64, 3, 1, 80, 80)))
    assert big.split_k == 1 and big.workspace_bytes == 0
    assert pl.m_tiles * pl.n_tiles < 152 and pl.split_k > 1
    assert pl.m_tiles * pl.n_tiles * pl.split_k <= 152 or pl.split_k == 1
    with pytest.raises(B.CbsError):   # FP32 only
        B.cbs_plan(make_desc(1, 64, 20, 20, 96, 3, 1, prec=B.CBS_TF32, in_layout=B.CBS_NHWC, force_variant=X3))
    # NCHW input: the same plan, the input read as given
    nchw = B.cbs_plan(make_desc(2, 64, 20, 20, 96, 3, 1, prec=B.CBS_FP32, in_layout=B.CBS_NCHW, force_variant=X3))
    assert nchw.variant == X3 and nchw.x_bytes == pl.x_bytes and nchw.split_k == pl.split_k
    assert nchw.workspace_bytes == pl.workspace_bytes
    # split-K on request: partial tiles and one counter per epilogue warp per tile
    sp = B.cbs_plan(desc_x3(2, spec, force_split_k=3))
    tiles = sp.m_tiles * sp.n_tiles
    assert sp.split_k == 3 and sp.grid_ctas == min(152, tiles * 3)
    assert sp.workspace_bytes == -(-tiles * 8 * 4 // 256) * 256 + tiles * 3 * 128 * sp.block_n * 4
    with pytest.raises(B.CbsError):   # more parts than pipeline stages
        B.cbs_plan(desc_x3(1, wl.LayerSpec(64, 64, 1, 1, 20, 20), force_split_k=8))


def test_automatic_choice(cuda_lib):
    """FP32 layers with NHWC input and channel counts that are multiples of
    8 take the 3xTF32 kernel on their own (the input bytes are then those of
    the CUDA-core kernel); otherwise the CUDA-core kernel (host-side, no GPU
    call)."""
    def variant(n, c_in, hw, c_out, k, stride, **kw):
        return B.cbs_plan(make_desc(n, c_in, hw, hw, c_out, k, stride, prec=B.CBS_FP32, **kw)).variant
    nhwc = dict(in_layout=B.CBS_NHWC)
    assert variant(16, 64, 80, 64, 3, 1, **nhwc) == X3               # 6400 x 16 pixels
    assert variant(1, 64, 80, 64, 3, 1, **nhwc) == X3                # 50 tiles
    assert variant(1, 128, 40, 128, 3, 1, **nhwc) == X3                # 13 pixel tiles: K parts fill the SMs
    assert variant(16, 64, 80, 64, 3, 1) == X3                        # NCHW input, 3x3
    assert variant(16, 64, 80, 64, 3, 2) == X3                        # NCHW input, stride 2
    assert variant(16, 64, 80, 64, 1, 1) == X3                        # NCHW input, 1x1 with 64 channels
    assert variant(16, 32, 80, 64, 1, 1) == B.CBS_VARIANT_SIMT_FP32   # NCHW input, 1x1 with 32 channels
    assert variant(16, 16, 80, 64, 3, 2) == B.CBS_VARIANT_SIMT_FP32   # NCHW input, 16 channels
    assert variant(16, 20, 80, 64, 3, 1, **nhwc) == B.CBS_VARIANT_SIMT_FP32   # 20 channels: would need padding
    assert variant(16, 3, 640, 16, 3, 2, **nhwc) == B.CBS_VARIANT_STEM
    p = B.cbs_plan(make_desc(16, 64, 80, 80, 64, 3, 1, prec=B.CBS_FP32, **nhwc))
    simt = B.cbs_plan(make_desc(16, 64, 80, 80, 64, 3, 1, prec=B.CBS_FP32, force_variant=B.CBS_VARIANT_SIMT_FP32,
                                **nhwc))
    assert p.x_bytes == simt.x_bytes and p.y_bytes == simt.y_bytes and p.desc.force_variant == -1
    two = B.cbs_plan(make_desc(16, 384, 40, 40, 128, 1, 1, prec=B.CBS_FP32, c_in_b=128, **nhwc))
    assert two.variant == X3 and two.x_b_bytes == 16 * 40 * 40 * 128 * 4


@pytest.mark.gpu
def test_automatic_choice_parity(cuda_lib):
    """A list layer at batch 16 with NHWC input through the default plan."""
    spec = wl.LAYER_LIST[3]
    x, p = wl.layer_inputs(spec, 16, layer_index=3)
    desc = make_desc(16, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad, prec=B.CBS_FP32,
                     in_layout=B.CBS_NHWC, out_layout=B.CBS_NCHW)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    assert layer.plan.variant == X3
    y = layer(layer.pack_input(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    for i in (0, 9):
        assert rel_l2(y[i:i + 1], ref_of(spec, x[i:i + 1], p)) <= TOL_FP32_REL_L2


@pytest.mark.gpu
@pytest.mark.parametrize("shape,split", [
    ((1, 256, 256, 3, 1, 20, 20), 8),      # the 20x20 list layer at batch 1: 4 x 3 tiles
    ((1, 128, 128, 3, 1, 40, 40), 4),      # the 40x40 list layer at batch 1
    ((1, 64, 96, 3, 2, 21, 19), 5),        # ragged pixels, parts of unequal length
    ((2, 384, 128, 1, 1, 12, 12), 3),      # 1x1, 2-D tile boxes
])
def test_split_k(cuda_lib, shape, split):
    """3xTF32 with K split over CTAs: each part's partial tile in the
    workspace, summed in order by the last arriving part."""
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=35)
    for out_layout in (B.CBS_NHWC, B.CBS_NCHW):
        y, layer = run_x3(spec, x, p, out_layout, force_split_k=split)
        assert layer.plan.split_k == split
        assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2
        # a second launch finds the counters back at zero
        y2 = layer(layer.pack_input(torch.from_numpy(x).cuda()))
        torch.cuda.synchronize()
        y2 = y2.cpu().numpy()
        y2 = nhwc_to_nchw(y2) if out_layout == B.CBS_NHWC else y2
        assert np.array_equal(y, y2)


@pytest.mark.gpu
def test_split_k_residual_two_inputs(cuda_lib):
    n, c_a, c_b, c_out, h = 1, 64, 64, 64, 10
    spec = wl.LayerSpec(c_a + c_b, c_out, 3, 1, h)
    x, p = wl.layer_inputs(spec, n, layer_index=36)
    r = np.random.default_rng(13).standard_normal((n, h, h, c_out)).astype(np.float32)
    desc = desc_x3(n, spec, activation=B.CBS_ACT_IDENTITY, residual=1, c_in_b=c_b, force_split_k=6)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    assert layer.plan.split_k == 6
    xa, xb = layer.pack_inputs(torch.from_numpy(np.ascontiguousarray(x[:, :c_a])).cuda(),
                               torch.from_numpy(np.ascontiguousarray(x[:, c_a:])).cuda())
    y = layer(xa, residual=torch.from_numpy(r).cuda(), x_b=xb)
    torch.cuda.synchronize()
    want = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1, act=B.CBS_ACT_IDENTITY,
                                  residual=np.ascontiguousarray(r.transpose(0, 3, 1, 2)))
    assert rel_l2(nhwc_to_nchw(y.cpu().numpy()), want) <= TOL_FP32_REL_L2


@pytest.mark.gpu
@pytest.mark.parametrize("ow_case", [(40, 48), (20, 32)])
def test_padded_rows_and_guard_bands_untouched(cuda_lib, ow_case):
    """NCHW output with a padded row pitch from the 3xTF32 kernel (unsplit
    and split): pad columns and a guard band after the buffer keep their
    sentinel."""
    size, pitch = ow_case
    spec = wl.LayerSpec(64, 32, 3, 1, size)
    x, p = wl.layer_inputs(spec, 2, layer_index=37)
    for split in (1, 3):
        desc = desc_x3(2, spec, out_layout=B.CBS_NCHW, out_row_stride=pitch, force_split_k=split)
        layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
        assert layer.plan.variant == X3 and layer.plan.split_k == split
        guard = 4096
        n_el = 2 * 32 * size * pitch
        buf = torch.full((n_el + guard,), float("nan"), dtype=torch.float32, device="cuda")
        sentinel_bits = buf[:1].view(torch.int32).item()
        y = buf[:n_el].view(2, 32, size, pitch)
        layer(layer.pack_input(torch.from_numpy(x).cuda()), y)
        torch.cuda.synchronize()
        host = buf.cpu()
        bits = host.view(torch.int32).numpy()
        yv = host[:n_el].view(2, 32, size, pitch).numpy()
        assert np.all(bits[n_el:] == sentinel_bits)
        assert np.all(yv[..., size:].view(np.int32) == sentinel_bits)
        assert rel_l2(yv[..., :size], ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.gpu
def test_empty_batch_is_a_noop(cuda_lib):
    spec = wl.LayerSpec(64, 64, 3, 1, 8)
    _, p = wl.layer_inputs(spec, 1)
    layer = FusedConvBnSilu(desc_x3(0, spec), p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    assert layer.plan.variant == X3
    y = layer(torch.empty((0, 8, 8, 64), dtype=torch.float32, device="cuda"),
              torch.empty((0, 8, 8, 64), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert y.numel() == 0


@pytest.mark.gpu
def test_automatic_split_matches_unsplit(cuda_lib):
    """A batch-1 list layer through the default plan (3xTF32, K in parts)
    against the same layer unsplit: both within the FP32 bar, and each
    launch of the split plan gives the same bits."""
    spec = wl.LAYER_LIST[10]
    x, p = wl.layer_inputs(spec, 1, layer_index=10)
    auto = FusedConvBnSilu(desc_x3(1, spec), p.w, p.gamma, p.beta, p.mean, p.var, p.eps, tuned=False)
    one = FusedConvBnSilu(desc_x3(1, spec, force_split_k=1), p.w, p.gamma, p.beta, p.mean, p.var, p.eps,
                          tuned=False)
    assert auto.plan.split_k > 1 and one.plan.split_k == 1
    xd = torch.from_numpy(x).cuda()
    ya = [nhwc_to_nchw(auto(auto.pack_input(xd)).cpu().numpy()) for _ in range(3)]
    y1 = nhwc_to_nchw(one(one.pack_input(xd)).cpu().numpy())
    want = ref_of(spec, x, p)
    assert rel_l2(ya[0], want) <= TOL_FP32_REL_L2 and rel_l2(y1, want) <= TOL_FP32_REL_L2
    for y in ya[1:]:
        assert np.array_equal(y.view(np.int32), ya[0].view(np.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("c_in,kw", [(512, {"force_split_k": 1, "force_block_n": 16}), (1024, {})])
def test_long_k_within_fp32_bar(cuda_lib, c_in, kw):
    """Long reductions (K = 4608 in one part, K = 9216 through the default
    plan): the tensor cores' accumulation error grows with the number of
    terms in one accumulator, so K is summed in chunks of at most 384 terms
    into separate accumulators and the chunks are added in FP32."""
    spec = wl.LayerSpec(c_in, 16, 3, 1, 12, 12)
    x, p = wl.layer_inputs(spec, 1, layer_index=41)
    y, layer = run_x3(spec, x, p, **kw)
    if "force_split_k" in kw:
        assert layer.plan.split_k == 1
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


def test_planner_matches_measured_choices(cuda_lib):
    """The 3xTF32 planner's N tile and K parts for the list layers (host-side,
    no GPU call) are the configurations measured fastest on GB300, or within a
    few percent of them: at batch 16 one N tile of 128 in 2 parts for the
    128->128 3x3 layer, 3 parts of 128 for 256->256 3x3; at batch 1 K parts
    that fill the SMs."""
    want = {
        16: {6: (128, 1), 7: (128, 2), 8: (256, 3), 10: (128, 3), 11: (128, 1)},
        1: {5: (64, 3), 8: (32, 4), 9: (32, 4), 11: (32, 2)},
    }
    for n, layers in want.items():
        for li, (bn, split) in layers.items():
            s = wl.LAYER_LIST[li]
            pl = B.cbs_plan(make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad, prec=B.CBS_FP32,
                                      in_layout=B.CBS_NHWC))
            assert pl.variant == X3 and (pl.block_n, pl.split_k) == (bn, split), (n, li, pl.block_n, pl.split_k)


def test_planner_keeps_accumulators_in_tmem(cuda_lib):
    """Every 3xTF32 plan over a spread of shapes: two accumulator buffers of
    (K-step chunks of at most 384 terms in the longest part) x N columns fit
    the 512 TMEM columns, parts never outnumber pipeline stages, and the
    grid never exceeds the SMs or the units."""
    rng = np.random.default_rng(5)
    def npow2(v):
        q = 1
        while q < v:
            q *= 2
        return q
    for _ in range(400):
        c_in = int(rng.choice([8, 16, 24, 32, 64, 96, 128, 256, 384, 512, 1024]))
        c_out = int(rng.choice([16, 32, 48, 64, 96, 128, 192, 256, 320]))
        k = int(rng.choice([1, 3, 5]))
        stride = int(rng.choice([1, 2]))
        hw = int(rng.integers(k, 90))
        n = int(rng.choice([1, 2, 16]))
        d = make_desc(n, c_in, hw, hw, c_out, k, stride, prec=B.CBS_FP32, in_layout=B.CBS_NHWC,
                      force_variant=X3)
        pl = B.cbs_plan(d)
        cb = pl.block_k
        ksteps = k * k * pl.c_in_pad // cb
        nst = ksteps // pl.k_group
        assert 1 <= pl.split_k <= nst
        unit = -(-nst // pl.split_k) * pl.k_group
        kpc = max(1, 384 // cb)
        chunks = -(-unit // kpc)
        assert 2 * chunks * npow2(pl.block_n) <= 512, (c_in, c_out, k, hw, n, pl.block_n, pl.split_k)
        units = pl.m_tiles * pl.n_tiles * pl.split_k
        assert pl.grid_ctas == min(152, units)


def run_nchw(spec, x, p, out_layout=B.CBS_NCHW, residual=None, **kw):
    """The layer with NCHW input: the 3xTF32 kernel, its converter warps
    reading x as given."""
    d = make_desc(x.shape[0], spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                  prec=B.CBS_FP32, in_layout=B.CBS_NCHW, out_layout=out_layout, **kw)
    layer = FusedConvBnSilu(d, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, tuned=False)
    xd = torch.from_numpy(x).cuda()
    y = layer(xd, residual=residual)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    return (nhwc_to_nchw(y) if out_layout == B.CBS_NHWC else y[..., :layer.plan.ow]), layer


@pytest.mark.gpu
@pytest.mark.parametrize("out_layout", [B.CBS_NCHW, B.CBS_NHWC])
@pytest.mark.parametrize("shape,kw", [
    ((1, 16, 32, 3, 2, 320, 320), {"force_variant": X3}),   # list layer 2: 16 channels, 64-byte blocks
    ((1, 64, 64, 3, 1, 80, 80), {}),                         # list layer 6 (chosen without forcing)
    ((1, 256, 256, 3, 1, 20, 20), {}),                       # list layer 11: K parts in the workspace too
    ((2, 24, 40, 3, 1, 17, 13), {"force_variant": X3}),      # ragged pixels and output channels
    ((2, 24, 40, 3, 2, 17, 13), {"force_variant": X3}),      # the same at stride 2
    ((1, 20, 16, 3, 1, 9, 11), {"force_variant": X3}),       # C_in 20: the gather zero-fills channels 20..23
    ((3, 64, 96, 1, 1, 9, 9), {"force_variant": X3}),        # 1x1 on request
    ((2, 32, 16, 3, 1, 1, 1), {"force_variant": X3}),        # 1x1 image: every tap but the centre in the padding
    ((3, 64, 40, 3, 2, 1, 2), {"force_variant": X3}),        # 1x2 image at stride 2
    ((1, 128, 128, 3, 1, 40, 40), {"force_variant": X3, "force_split_k": 3}),   # forced K parts
])
def test_fp32_nchw_input_on_tensor_cores(cuda_lib, out_layout, shape, kw):
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=34)
    y, layer = run_nchw(spec, x, p, out_layout, **kw)
    pl = layer.plan
    assert pl.variant == X3
    assert pl.x_bytes == x.nbytes
    assert (pl.workspace_bytes > 0) == (pl.split_k > 1)
    e = rel_l2(y, ref_of(spec, x, p))
    assert e <= TOL_FP32_REL_L2, e
    y2, _ = run_nchw(spec, x, p, out_layout, **kw)
    assert np.array_equal(y, y2)


@pytest.mark.gpu
def test_fp32_nchw_input_padded_rows_and_residual(cuda_lib):
    """NCHW in and out with a padded output row pitch, the identity
    activation and a residual: columns past OW stay untouched."""
    spec = wl.LayerSpec(32, 48, 3, 1, 21, 21)
    x, p = wl.layer_inputs(spec, 2, layer_index=35)
    r = np.random.default_rng(6).standard_normal((2, 48, 21, 21)).astype(np.float32)
    stride = 32
    rp = np.zeros((2, 48, 21, stride), np.float32)
    rp[..., :21] = r
    d = make_desc(2, 32, 21, 21, 48, 3, 1, prec=B.CBS_FP32, in_layout=B.CBS_NCHW, out_layout=B.CBS_NCHW,
                  out_row_stride=stride, activation=B.CBS_ACT_IDENTITY, residual=1)
    layer = FusedConvBnSilu(d, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, tuned=False)
    assert layer.plan.variant == X3
    y = torch.full((2, 48, 21, stride), 7.0, device="cuda")
    layer(torch.from_numpy(x).cuda(), y, residual=torch.from_numpy(rp).cuda())
    y = y.cpu().numpy()
    want = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1, act=1, residual=r)
    assert rel_l2(y[..., :21], want) <= TOL_FP32_REL_L2
    assert np.all(y[..., 21:] == 7.0)


@pytest.mark.gpu
@pytest.mark.parametrize("i", [5, 10])
def test_fp32_nchw_input_batch16(cuda_lib, i):
    """List layers 6 and 11 at batch 16 with NCHW input, every image against
    the oracle: the converter warps' gather over several tiles per persistent
    CTA (layer 6: 800 tiles) and over K parts (layer 11), images crossed
    inside tiles."""
    spec = wl.LAYER_LIST[i]
    x, p = wl.layer_inputs(spec, 16, layer_index=i)
    y, layer = run_nchw(spec, x, p)
    pl = layer.plan
    assert pl.variant == X3 and (pl.m_tiles * pl.n_tiles > 152 or pl.split_k > 1)
    e = rel_l2(y, ref_of(spec, x, p))
    assert e <= TOL_FP32_REL_L2, e


FLAT = {"force_variant": X3, "force_window": 1}


@pytest.mark.gpu
@pytest.mark.parametrize("out_layout", [B.CBS_NCHW, B.CBS_NHWC])
@pytest.mark.parametrize("shape,kw", [
    ((1, 64, 64, 1, 1, 80, 80), FLAT),                       # list layer 5: 1x1
    ((1, 64, 64, 3, 1, 80, 80), FLAT),                       # list layer 6
    ((1, 128, 128, 3, 1, 40, 40), FLAT),                     # list layer 8
    ((1, 256, 256, 1, 1, 20, 20), FLAT),                     # list layer 10
    ((1, 256, 256, 3, 1, 20, 20), FLAT),                     # list layer 11: K parts in the workspace
    ((1, 384, 128, 1, 1, 40, 40), FLAT),                     # list layer 12
    ((1, 20, 16, 3, 1, 12, 12), FLAT),                       # C_in 20: 8-channel blocks, channels 20..23 zero
    ((2, 24, 40, 3, 1, 16, 16), FLAT),                       # batch 2, two whole tiles per image
    ((1, 32, 48, 5, 1, 20, 24), FLAT),                       # 5x5, pad 2
    ((1, 32, 16, 7, 1, 12, 8), FLAT),                        # 7x7, pad 3: column offsets -3..3
    ((1, 64, 64, 3, 1, 4, 4), FLAT),                         # 4x4 image: one partial tile, rows in the fill
    ((1, 32, 40, 3, 1, 8, 100), FLAT),                       # rows of 100: tiles end mid-row
    ((1, 128, 128, 3, 1, 40, 40), dict(FLAT, force_split_k=3)),   # forced K parts
])
def test_fp32_nchw_flat_boxes(cuda_lib, out_layout, shape, kw):
    """NCHW input in flat TMA boxes (stride-1 layers with k = 2 pad + 1):
    every filter row's pixels as one box per K step, the wrapped columns
    zeroed by the converters."""
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=36)
    y, layer = run_nchw(spec, x, p, out_layout, **kw)
    pl = layer.plan
    assert pl.variant == X3 and pl.window == 1 and pl.threads == 608
    assert pl.x_bytes == x.nbytes
    e = rel_l2(y, ref_of(spec, x, p))
    assert e <= TOL_FP32_REL_L2, e
    y2, _ = run_nchw(spec, x, p, out_layout, **kw)
    assert np.array_equal(y, y2)
    # the same numbers as the gather, up to the order of the partial sums
    yg, lg = run_nchw(spec, x, p, out_layout, **{kk: v for kk, v in kw.items() if kk != "force_window"})
    assert lg.plan.window == 0
    assert rel_l2(y, yg) <= TOL_FP32_REL_L2


@pytest.mark.gpu
def test_fp32_nchw_flat_boxes_padded_rows_and_residual(cuda_lib):
    """Flat boxes with a padded NCHW output pitch, the identity activation
    and a residual: columns past OW stay untouched."""
    spec = wl.LayerSpec(32, 48, 3, 1, 20, 20)
    x, p = wl.layer_inputs(spec, 1, layer_index=37)
    r = np.random.default_rng(7).standard_normal((1, 48, 20, 20)).astype(np.float32)
    stride = 24
    rp = np.zeros((1, 48, 20, stride), np.float32)
    rp[..., :20] = r
    d = make_desc(1, 32, 20, 20, 48, 3, 1, prec=B.CBS_FP32, in_layout=B.CBS_NCHW, out_layout=B.CBS_NCHW,
                  out_row_stride=stride, activation=B.CBS_ACT_IDENTITY, residual=1, **FLAT)
    layer = FusedConvBnSilu(d, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, tuned=False)
    assert layer.plan.variant == X3 and layer.plan.window == 1
    y = torch.full((1, 48, 20, stride), 7.0, device="cuda")
    layer(torch.from_numpy(x).cuda(), y, residual=torch.from_numpy(rp).cuda())
    y = y.cpu().numpy()
    want = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1, act=1, residual=r)
    assert rel_l2(y[..., :20], want) <= TOL_FP32_REL_L2
    assert np.all(y[..., 20:] == 7.0)


@pytest.mark.gpu
def test_fp32_nchw_flat_boxes_batch16(cuda_lib):
    """List layer 6 at batch 16 in flat boxes, every image against the
    oracle: 50 whole tiles per image, persistent CTAs walking several."""
    spec = wl.LAYER_LIST[5]
    x, p = wl.layer_inputs(spec, 16, layer_index=5)
    y, layer = run_nchw(spec, x, p, **FLAT)
    assert layer.plan.window == 1 and layer.plan.m_tiles == 800
    e = rel_l2(y, ref_of(spec, x, p))
    assert e <= TOL_FP32_REL_L2, e


def test_nchw_flat_box_rules(cuda_lib):
    """Host-side: flat boxes only where every filter row of a tile is one
    aligned run of an NCHW channel row; a box lands over its K step's A
    tiles, so a stage (one K step) is the size of the gather's K step."""
    def plan(n, c_in, h, w, k, stride, pad=None, **kw):
        return B.cbs_plan(make_desc(n, c_in, h, w, 64, k, stride, pad, prec=B.CBS_FP32, in_layout=B.CBS_NCHW,
                                    **dict(FLAT, **kw)))
    pl = plan(1, 64, 80, 80, 3, 1)
    assert pl.window == 1 and pl.threads == 608
    gather = B.cbs_plan(make_desc(1, 64, 80, 80, 64, 3, 1, prec=B.CBS_FP32, in_layout=B.CBS_NCHW,
                                  force_variant=X3, force_split_k=pl.split_k, force_block_n=pl.block_n))
    assert gather.window == 0
    def kstep_bytes(q):   # shared memory = 1 KB alignment + stages x K steps + barriers
        return (q.smem_bytes - 1024 - 8 * (3 * q.stages + 5) - 16) // (q.stages * q.k_group)
    assert pl.k_group == 1 and kstep_bytes(pl) == kstep_bytes(gather)
    assert kstep_bytes(pl) >= 136 * 32 * 4 + 2 * 64 * 128   # the box and the two weight tiles
    assert plan(2, 64, 16, 16, 3, 1).window == 1            # 256 pixels: two whole tiles per image
    for bad in (dict(n=1, c_in=64, h=80, w=80, k=3, stride=2),     # stride 2
                dict(n=1, c_in=64, h=80, w=80, k=3, stride=1, pad=0),   # output grid smaller than the input
                dict(n=1, c_in=64, h=21, w=21, k=3, stride=1),     # W not a multiple of 4
                dict(n=2, c_in=64, h=20, w=20, k=3, stride=1),     # 400 pixels: tiles would span images
                dict(n=1, c_in=64, h=20, w=20, k=9, stride=1)):    # pad 4: column offsets past the box
        with pytest.raises(B.CbsError) as ei:
            plan(**bad)
        assert ei.value.status == B.CBS_ERR_UNSUPPORTED
    with pytest.raises(B.CbsError) as ei:
        B.cbs_plan(make_desc(1, 64, 80, 80, 64, 3, 1, prec=B.CBS_FP32, in_layout=B.CBS_NHWC, **FLAT))
    assert ei.value.status == B.CBS_ERR_UNSUPPORTED


def test_nchw_mode_launch_shape(cuda_lib):
    """Host-side: the NCHW mode runs 608 threads (eight converter warps), the
    NHWC kernel 480 (four); both use the same tiles and shared memory."""
    kw = dict(prec=B.CBS_FP32, force_variant=X3)
    nchw = B.cbs_plan(make_desc(2, 64, 20, 20, 96, 3, 1, in_layout=B.CBS_NCHW, **kw))
    nhwc = B.cbs_plan(make_desc(2, 64, 20, 20, 96, 3, 1, in_layout=B.CBS_NHWC, **kw))
    assert (nchw.threads, nhwc.threads) == (608, 480)
    assert (nchw.block_m, nchw.block_n, nchw.stages, nchw.split_k, nchw.smem_bytes) == \
        (nhwc.block_m, nhwc.block_n, nhwc.stages, nhwc.split_k, nhwc.smem_bytes)
