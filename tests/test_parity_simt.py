"""GPU parity of the FP32 CUDA-core path against the CPU oracle.

Bar: relative L2 <= 1e-5 over the whole output, element by element on the
same seeded inputs.  Covers the single 40x40 layer, every layer of the
twelve-layer list at batch 1 and full size, forced tiles and split-K,
NHWC, ragged and degenerate shapes, padded output rows with canaries, and
run-to-run determinism."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import TOL_FP32_REL_L2, max_abs, nchw_to_nhwc, nhwc_to_nchw, rel_l2

pytestmark = pytest.mark.gpu


def run_simt(spec, x, p, in_layout=B.CBS_NCHW, out_layout=B.CBS_NCHW, **kw):
    n = x.shape[0]
    if in_layout == B.CBS_NHWC:   # FP32 NHWC layers would otherwise take the 3xTF32 kernel
        kw.setdefault("force_variant", B.CBS_VARIANT_SIMT_FP32)
    desc = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                     prec=B.CBS_FP32, in_layout=in_layout, out_layout=out_layout, **kw)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xin = x if in_layout == B.CBS_NCHW else nchw_to_nhwc(x)
    xd = torch.from_numpy(np.ascontiguousarray(xin)).cuda()
    y = layer(xd)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    if out_layout == B.CBS_NHWC:
        y = nhwc_to_nchw(y)
    return y, layer


def ref_of(spec, x, p):
    return oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad)


def test_single_layer_40x40(cuda_lib):
    spec = wl.SINGLE_LAYER
    x, p = wl.layer_inputs(spec, 1)
    y, layer = run_simt(spec, x, p)
    ref = ref_of(spec, x, p)
    assert y.shape == ref.shape
    assert rel_l2(y, ref) <= TOL_FP32_REL_L2
    assert max_abs(y, ref) < 1e-4


@pytest.mark.parametrize("i", range(len(wl.LAYER_LIST)))
def test_layer_list_batch1(cuda_lib, i):
    spec = wl.LAYER_LIST[i]
    x, p = wl.layer_inputs(spec, 1, layer_index=i)
    y, layer = run_simt(spec, x, p)
    ref = ref_of(spec, x, p)
    err = rel_l2(y, ref)
    assert err <= TOL_FP32_REL_L2, (i, err, layer.plan.block_m, layer.plan.block_n, layer.plan.split_k)


@pytest.mark.parametrize("split", [1, 2, 3, 7, 16])
def test_forced_split_k(cuda_lib, split):
    spec = wl.LayerSpec(256, 256, 3, 1, 20)
    x, p = wl.layer_inputs(spec, 1, layer_index=10)
    y, layer = run_simt(spec, x, p, force_split_k=split)
    assert layer.plan.split_k == split
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("bn", [16, 32, 64, 128])
def test_forced_tiles(cuda_lib, bn):
    spec = wl.LayerSpec(32, 48, 3, 2, 33)
    x, p = wl.layer_inputs(spec, 2, layer_index=4)
    y, layer = run_simt(spec, x, p, force_block_n=bn)
    assert layer.plan.block_n == bn
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("bm,bn,split", [(128, 128, 1), (128, 128, 4), (128, 64, 2), (256, 16, 3)])
@pytest.mark.parametrize("layouts", [(B.CBS_NCHW, B.CBS_NCHW), (B.CBS_NHWC, B.CBS_NHWC)])
def test_forced_large_tiles(cuda_lib, bm, bn, split, layouts):
    """Tiles whose shared memory exceeds 48 KB (128x128: the staged output
    tile alone is 67 KB) run with the raised dynamic shared-memory ceiling."""
    spec = wl.LayerSpec(64, 160, 3, 1, 21)
    x, p = wl.layer_inputs(spec, 2, layer_index=5)
    y, layer = run_simt(spec, x, p, in_layout=layouts[0], out_layout=layouts[1], force_block_m=bm,
                        force_block_n=bn, force_split_k=split)
    assert (layer.plan.block_m, layer.plan.block_n, layer.plan.split_k) == (bm, bn, split)
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("layouts", [(B.CBS_NHWC, B.CBS_NHWC), (B.CBS_NCHW, B.CBS_NHWC), (B.CBS_NHWC, B.CBS_NCHW)])
def test_layouts(cuda_lib, layouts):
    spec = wl.LayerSpec(24, 40, 3, 1, 17)
    x, p = wl.layer_inputs(spec, 2, layer_index=6)
    y, _ = run_simt(spec, x, p, in_layout=layouts[0], out_layout=layouts[1])
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("shape", [
    (3, 5, 7, 3, 2, 13),    # ragged everything, stride 2
    (1, 1, 1, 3, 1, 1),     # 1x1 image, 3x3 filter, one channel
    (2, 3, 9, 1, 1, 11),    # 1x1 conv
    (1, 7, 1, 3, 1, 6),     # one output channel
    (5, 130, 129, 3, 1, 5), # channels just past tile sizes
])
def test_ragged_and_degenerate(cuda_lib, shape):
    n, c_in, c_out, k, stride, h = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=7)
    y, _ = run_simt(spec, x, p)
    assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("variant", [B.CBS_VARIANT_SIMT_FP32, B.CBS_VARIANT_STEM])
@pytest.mark.parametrize("layouts", [(B.CBS_NCHW, B.CBS_NCHW), (B.CBS_NHWC, B.CBS_NHWC), (B.CBS_NCHW, B.CBS_NHWC)])
def test_small_channel_layers_both_kernels(cuda_lib, variant, layouts):
    """The stem shape through the implicit GEMM and through the direct
    kernel, with ragged sizes and both layouts."""
    for shape in ((2, 3, 16, 3, 2, 37), (1, 4, 24, 3, 1, 19), (3, 1, 5, 1, 1, 9), (1, 2, 64, 5, 2, 23),
                  (1, 4, 64, 7, 2, 29)):  # 7x7 x 4 x 64 weights: 49 KB of shared memory
        n, c_in, c_out, k, stride, h = shape
        spec = wl.LayerSpec(c_in, c_out, k, stride, h)
        x, p = wl.layer_inputs(spec, n, layer_index=12)
        y, layer = run_simt(spec, x, p, in_layout=layouts[0], out_layout=layouts[1], force_variant=variant)
        assert layer.plan.variant == variant
        assert rel_l2(y, ref_of(spec, x, p)) <= TOL_FP32_REL_L2, (shape, variant)


def test_empty_batch_is_a_noop(cuda_lib):
    spec = wl.LayerSpec(8, 8, 3, 1, 6)
    _, p = wl.layer_inputs(spec, 1)
    desc = make_desc(0, 8, 6, 6, 8, 3, 1)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    x = torch.empty((0, 8, 6, 6), dtype=torch.float32, device="cuda")
    y = layer(x, torch.empty((0, 8, 6, 6), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert y.numel() == 0


@pytest.mark.parametrize("ow_case", [(40, 48), (20, 32), (40, 40)])
def test_padded_rows_and_guard_bands_untouched(cuda_lib, ow_case):
    """Output rows with a padded pitch: pad columns and a guard band after
    the buffer keep their sentinel (the failure page 1 describes)."""
    size, pitch = ow_case
    spec = wl.LayerSpec(16, 32, 3, 1, size)
    x, p = wl.layer_inputs(spec, 2, layer_index=1)
    desc = make_desc(2, 16, size, size, 32, 3, 1, out_row_stride=pitch)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    guard = 4096
    n_el = 2 * 32 * size * pitch
    buf = torch.full((n_el + guard,), float("nan"), dtype=torch.float32, device="cuda")
    sentinel_bits = buf[:1].view(torch.int32).item()
    y = buf[:n_el].view(2, 32, size, pitch)
    layer(torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    host = buf.cpu()
    bits = host.view(torch.int32).numpy()
    yv = host[:n_el].view(2, 32, size, pitch).numpy()
    assert np.all(bits[n_el:] == sentinel_bits)
    assert np.all(yv[..., size:].view(np.int32) == sentinel_bits)
    assert rel_l2(yv[..., :size], ref_of(spec, x, p)) <= TOL_FP32_REL_L2


def test_split_k_is_deterministic_and_reusable(cuda_lib):
    spec = wl.LayerSpec(128, 256, 3, 2, 40)
    x, p = wl.layer_inputs(spec, 1, layer_index=8)
    desc = make_desc(1, 128, 40, 40, 256, 3, 2, force_split_k=6)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xd = torch.from_numpy(x).cuda()
    outs = [layer(xd).cpu().numpy() for _ in range(4)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.int32), outs[0].view(np.int32))
    assert rel_l2(outs[0], ref_of(spec, x, p)) <= TOL_FP32_REL_L2


def test_no_timeout_reported(cuda_lib):
    assert B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream) == B.CBS_OK
