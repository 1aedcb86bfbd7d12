"""GPU parity of the INT8 path against the CPU oracle: bit-exact.

Each stage is compared byte for byte with the oracle on the same seeded
inputs: the activation quantiser (cbs_pack_input), the quantising fold
(int8 codes, int32 bias, m_c), and the fused INT8 layer (integer sums,
int32 bias, SiLU in float with the specified exp, round half to even)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import nhwc_to_nchw

pytestmark = pytest.mark.gpu

SCALES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "int8_scales.json")))
S_X = float(wl.S_X_INT8)


def build(spec, n, p, out_layout=B.CBS_NHWC, **kw):
    desc = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                     prec=B.CBS_INT8, in_layout=B.CBS_NHWC, out_layout=out_layout, **kw)
    return FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=S_X)


def gpu_packed_codes(layer, spec):
    """The fold's packed weights back in OIHW int8 (bf16 codes -> int)."""
    c_pad = layer.plan.c_in_pad
    wb = layer.w_packed.view(torch.bfloat16).float().cpu().numpy()
    wb = wb.reshape(spec.c_out, spec.k, spec.k, c_pad)
    assert np.all(wb[..., spec.c_in:] == 0)
    assert np.all(wb == np.round(wb))
    return wb[..., :spec.c_in].transpose(0, 3, 1, 2).astype(np.int8)


def run_layer(spec, x, p, s_y, out_layout=B.CBS_NHWC, **kw):
    n = x.shape[0]
    layer = build(spec, n, p, out_layout=out_layout, **kw)
    qx = layer.pack_input(torch.from_numpy(x).cuda())
    y = layer(qx, s_y=s_y)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    if out_layout == B.CBS_NHWC:
        y = nhwc_to_nchw(y)
    return layer, qx.cpu().numpy(), y


def oracle_layer(spec, x, p, s_y):
    q_x = oracle.quantize_act(x, S_X)
    q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, S_X)
    q_y = oracle.conv_i8(q_x, q_w, bias, m_c, s_y, spec.stride, spec.pad)
    return q_x, q_w, bias, m_c, q_y


def assert_bit_exact(spec, x, p, s_y, what="", **kw):
    layer, qx_gpu, y_gpu = run_layer(spec, x, p, s_y, **kw)
    q_x, q_w, bias, m_c, q_y = oracle_layer(spec, x, p, s_y)
    c_pad = layer.plan.c_in_pad
    qx_gpu = qx_gpu.reshape(x.shape[0], spec.h, spec.width, c_pad)
    assert np.all(qx_gpu[..., spec.c_in:] == 0)
    assert np.array_equal(nhwc_to_nchw(qx_gpu[..., :spec.c_in]), q_x), ("quantised input", what)
    assert np.array_equal(gpu_packed_codes(layer, spec), q_w), ("weight codes", what)
    assert np.array_equal(layer.bias.view(torch.int32).cpu().numpy(), bias), ("int32 bias", what)
    assert np.array_equal(layer.m_c.cpu().numpy().view(np.int32), m_c.view(np.int32)), ("m_c", what)
    mism = int(np.count_nonzero(y_gpu != q_y))
    assert mism == 0, (what, mism, y_gpu.size)
    return y_gpu


def test_single_layer(cuda_lib):
    spec = wl.SINGLE_LAYER
    x, p = wl.layer_inputs(spec, 1)
    y = assert_bit_exact(spec, x, p, SCALES["single_layer"])
    assert len(np.unique(y)) > 50  # the scale puts outputs across the code range


@pytest.mark.parametrize("i", range(len(wl.LAYER_LIST)))
def test_layer_list_batch1(cuda_lib, i):
    spec = wl.LAYER_LIST[i]
    x, p = wl.layer_inputs(spec, 1, layer_index=i)
    assert_bit_exact(spec, x, p, SCALES["layer_list"][i], i)


@pytest.mark.parametrize("i", range(len(wl.LAYER_LIST)))
def test_batch16_layer_list(cuda_lib, i):
    """The INT8 config: every list layer at batch 16, all 16 images bit for
    bit against the oracle, with the quantiser, the fold and the layer each
    compared."""
    spec = wl.LAYER_LIST[i]
    x, p = wl.layer_inputs(spec, 16, layer_index=i)
    y = assert_bit_exact(spec, x, p, SCALES["layer_list"][i], i)
    assert y.shape[0] == 16


@pytest.mark.parametrize("shape", [
    (3, 16, 48, 3, 2, 13),     # ragged pixels, stride 2
    (2, 32, 16, 1, 1, 11),     # 1x1, tail tile
    (1, 64, 272, 3, 1, 6),     # two N tiles, second ragged
    (2, 48, 32, 3, 1, 9),      # C_in = 48: 16-channel K steps
    (1, 3, 16, 3, 2, 34),      # C_in = 3 padded to 16
    (1, 256, 64, 3, 1, 5),     # K = 2304: three exact-sum chunks
    (1, 384, 32, 1, 1, 7),     # 1x1 with 384 channels
])
def test_ragged(cuda_lib, shape):
    n, c_in, c_out, k, stride, h = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=11)
    assert_bit_exact(spec, x, p, 0.05, shape)



@pytest.mark.parametrize("kg", [1, 2, 3, 4])
@pytest.mark.parametrize("shape,bn", [
    ((1, 128, 64, 3, 1, 9), 64),     # 18 K steps, two exact-sum chunks: a 3-step stage spans the boundary
    ((1, 256, 96, 3, 1, 5), 48),     # 36 K steps, three chunks, two N tiles
    ((2, 32, 32, 3, 2, 13), 32),     # 9 K steps of 32 channels
])
def test_k_steps_per_stage(cuda_lib, shape, bn, kg):
    """Several K steps per pipeline stage, including stages that straddle an
    exact-sum chunk boundary (each K step picks its chunk's accumulator)."""
    n, c_in, c_out, k, stride, h = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=14)
    ksteps = k * k * (c_in // (64 if c_in % 64 == 0 else 32))
    if ksteps % kg:
        with pytest.raises(B.CbsError):
            build(spec, n, p, force_k_group=kg, force_block_n=bn)
        return
    try:
        layer = build(spec, n, p, force_k_group=kg, force_block_n=bn)
    except B.CbsError as e:   # two stages of kg K steps exceed shared memory
        assert e.status == B.CBS_ERR_UNSUPPORTED and kg == 4
        return
    assert layer.plan.k_group == kg and layer.plan.block_n == bn
    assert_bit_exact(spec, x, p, 0.05, (shape, kg), force_k_group=kg, force_block_n=bn)

def test_nchw_output(cuda_lib):
    spec = wl.LayerSpec(32, 48, 3, 1, 10)
    x, p = wl.layer_inputs(spec, 2, layer_index=2)
    assert_bit_exact(spec, x, p, 0.06, out_layout=B.CBS_NCHW)


@pytest.mark.parametrize("s_y", [1e-4, 10.0])
def test_saturation_and_underflow(cuda_lib, s_y):
    """Tiny s_y saturates most outputs at -128/127; a huge one rounds them to 0."""
    spec = wl.LayerSpec(16, 32, 3, 1, 12)
    x, p = wl.layer_inputs(spec, 1, layer_index=4)
    y = assert_bit_exact(spec, x, p, s_y)
    if s_y < 1:
        assert (y == 127).mean() > 0.3
    else:
        assert (y == 0).mean() > 0.9


def test_no_timeout_reported(cuda_lib):
    assert B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream) == B.CBS_OK


@pytest.mark.parametrize("shape,z", [
    ((2, 3, 16, 3, 2, 34), (-61, 17)),       # stem (direct kernel), pixel windows leave the image at every edge
    ((1, 4, 32, 7, 2, 23), (90, -128)),      # 7x7 stem: many out-of-image taps
    ((2, 16, 32, 3, 2, 21), (-128, 127)),    # tensor cores, stride 2, ragged pixel tiles
    ((1, 32, 48, 3, 1, 9), (45, -100)),      # small image: most windows touch a border
    ((2, 48, 64, 1, 1, 11), (-20, 3)),       # 1x1: no padding, only the zero point itself
    ((1, 64, 32, 5, 1, 13), (127, 0)),       # 5x5, output symmetric
])
def test_asymmetric_zero_points(cuda_lib, shape, z):
    """Asymmetric activations (input and output zero points) bit for bit
    against the oracle: the quantiser, the fold's bias, and the layer, for
    the direct small-channel kernel and the tensor-core kernel."""
    n, c_in, c_out, k, stride, h = shape
    z_x, z_y = z
    spec = wl.LayerSpec(c_in, c_out, k, stride, h)
    x, p = wl.layer_inputs(spec, n, layer_index=13)
    x = (x / (1 + np.exp(-x)) * 3).astype(np.float32)   # mostly positive, like activations after SiLU
    y32 = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, stride, spec.pad)
    s_y = float(np.float32(np.abs(y32).max() / 200))
    desc = make_desc(n, c_in, h, h, c_out, k, stride, spec.pad, prec=B.CBS_INT8, in_layout=B.CBS_NHWC,
                     out_layout=B.CBS_NHWC, zero_point_x=z_x, zero_point_y=z_y)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=S_X)
    qx = layer.pack_input(torch.from_numpy(x).cuda())
    y = nhwc_to_nchw(layer(qx, s_y=s_y).cpu().numpy())
    q_x = oracle.quantize_act(x, S_X, z_x)
    q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, S_X)
    want = oracle.conv_i8(q_x, q_w, bias, m_c, s_y, stride, spec.pad, z_x=z_x, z_y=z_y)
    c_pad = layer.plan.c_in_pad
    qg = qx.cpu().numpy().reshape(n, h, h, c_pad)
    assert np.array_equal(nhwc_to_nchw(qg[..., :c_in]), q_x) and np.all(qg[..., c_in:] == 0)
    qsum = q_w.astype(np.int64).reshape(c_out, -1).sum(axis=1)
    want_bias = ((bias.astype(np.int64) - z_x * qsum + 2**31) % 2**32 - 2**31).astype(np.int32)
    assert np.array_equal(layer.bias.view(torch.int32).cpu().numpy(), want_bias)
    mism = int(np.count_nonzero(y != want))
    assert mism == 0, (layer.plan.variant, mism, y.size)
    if abs(z_y) < 100:   # (an output zero point at an end of the code range saturates half the outputs)
        assert len(np.unique(y)) > 20


@pytest.mark.parametrize("out_layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("shape,z", [
    ((2, 3, 16, 3, 2, 38, 38), (0, 0)),        # 3x3 s2, even width: pixel-pair loads
    ((2, 3, 16, 3, 2, 37, 37), (-40, 9)),      # odd width: one load per tap
    ((1, 4, 32, 3, 1, 19, 19), (17, -3)),      # stride 1
    ((3, 1, 48, 1, 1, 9, 9), (5, 60)),         # 1x1, C_out 48: 4 CTAs per SM (TMEM)
    ((1, 2, 64, 3, 2, 50, 34), (-128, 127)),   # C_out 64, non-square, zero points at the ends
    ((1, 3, 20, 3, 2, 22, 22), (3, -7)),       # C_out 20: per-channel stores
    ((4, 3, 16, 3, 2, 160, 160), (-20, -100)), # 1600 tiles: several per persistent CTA
])
def test_tensor_core_stem_i8(cuda_lib, out_layout, shape, z):
    """INT8 layers with at most 4 input channels and k <= 3 run on the
    tensor-core stem: bit for bit against the oracle."""
    n, c_in, c_out, k, stride, h, w = shape
    z_x, z_y = z
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=19)
    y32 = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, stride, spec.pad)
    s_y = float(np.float32(np.abs(y32).max() / 110))
    desc = make_desc(n, c_in, h, w, c_out, k, stride, spec.pad, prec=B.CBS_INT8, in_layout=B.CBS_NHWC,
                     out_layout=out_layout, zero_point_x=z_x, zero_point_y=z_y)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=S_X)
    pl = layer.plan
    assert pl.variant == B.CBS_VARIANT_STEM and pl.block_m == 128 and pl.threads == 256
    y = layer(layer.pack_input(torch.from_numpy(x).cuda()), s_y=s_y).cpu().numpy()
    if out_layout == B.CBS_NHWC:
        y = nhwc_to_nchw(y)
    q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, S_X)
    want = oracle.conv_i8(oracle.quantize_act(x, S_X, z_x), q_w, bias, m_c, s_y, stride, spec.pad,
                          z_x=z_x, z_y=z_y)
    assert int(np.count_nonzero(y != want)) == 0, shape
