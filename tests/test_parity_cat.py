"""GPU parity of two-input layers: conv over concat(x, x_b) along channels,
read straight from the two tensors (page 1, "Improvements" #6: channel_cat
fused into the convolution's input loads).  The oracle convolves the
concatenated array.  Covered: the CUDA-core implicit GEMM in both layouts
(with split-K), the TF32/BF16 tensor-core kernel on each A path (2-D tiles
for 1x1, im2col boxes, windowed A) with the channel block boundary at the
junction of the two inputs and a second input padded with zero channels, and
the INT8 kernel (bit-exact, symmetric and with zero points).  Bars as for the
one-input layer."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import TOL_FP32_REL_L2, check_tc, nhwc_to_nchw, rel_l2, tc_refs

pytestmark = pytest.mark.gpu

PRECS = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16}


def run_cat(n, c_a, c_b, c_out, k, stride, h, w, prec, in_layout, out_layout, **kw):
    spec = wl.LayerSpec(c_a + c_b, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=21)
    xa, xb = np.ascontiguousarray(x[:, :c_a]), np.ascontiguousarray(x[:, c_a:])
    desc = make_desc(n, c_a + c_b, h, w, c_out, k, stride, spec.pad, prec=PRECS[prec], in_layout=in_layout,
                     out_layout=out_layout, c_in_b=c_b, **kw)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    assert layer.plan.desc.c_in_b == c_b
    pa, pb = layer.pack_inputs(torch.from_numpy(xa).cuda(), torch.from_numpy(xb).cuda())
    assert pa.numel() * pa.element_size() == layer.plan.x_bytes
    assert pb.numel() * pb.element_size() == layer.plan.x_b_bytes
    y = layer(pa, x_b=pb)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy()
    if out_layout == B.CBS_NHWC:
        got = nhwc_to_nchw(got)
    else:
        got = got[..., : spec.ow]
    return got, x, p, spec, layer


def ref(x, p, spec):
    return oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad)


@pytest.mark.parametrize("layouts", [(B.CBS_NCHW, B.CBS_NCHW), (B.CBS_NHWC, B.CBS_NHWC), (B.CBS_NHWC, B.CBS_NCHW)])
@pytest.mark.parametrize("shape", [
    (2, 256, 128, 128, 1, 1, 20, 20),    # the neck's 384->128 1x1 layer at 20x20
    (1, 32, 16, 64, 3, 1, 20, 20),       # 3x3
    (1, 24, 16, 40, 3, 2, 17, 13),       # stride 2, ragged everything
    (2, 5, 3, 16, 3, 1, 9, 9),           # few channels on each side
])
def test_cuda_core_two_inputs(cuda_lib, layouts, shape):
    n, c_a, c_b, c_out, k, stride, h, w = shape
    got, x, p, spec, layer = run_cat(n, c_a, c_b, c_out, k, stride, h, w, "fp32", *layouts,
                                     force_variant=B.CBS_VARIANT_SIMT_FP32)
    assert layer.plan.variant == B.CBS_VARIANT_SIMT_FP32
    assert rel_l2(got, ref(x, p, spec)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("split", [2, 5])
def test_cuda_core_two_inputs_split_k(cuda_lib, split):
    """K partitions that start inside either input."""
    got, x, p, spec, layer = run_cat(1, 96, 64, 64, 3, 1, 12, 12, "fp32", B.CBS_NCHW, B.CBS_NCHW,
                                     force_split_k=split)
    assert layer.plan.split_k == split
    assert rel_l2(got, ref(x, p, spec)) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("case", [
    ((2, 256, 128, 128, 1, 1, 20, 20), {}),                   # 1x1 stride 1: 2-D tile boxes
    ((1, 64, 64, 64, 3, 1, 20, 20), {}),                      # im2col boxes
    ((1, 64, 32, 96, 3, 2, 21, 19), {}),                      # stride 2, ragged pixels
    ((1, 48, 8, 32, 3, 1, 11, 11), {}),                       # second input padded with zero channels
    ((2, 64, 64, 64, 3, 1, 16, 16), {"force_window": 1}),     # windowed A, one window per channel block
    ((2, 64, 64, 64, 3, 1, 16, 16), {"force_k_group": 3, "force_b_resident": 1}),
])
def test_tensor_core_two_inputs(cuda_lib, prec, case):
    (n, c_a, c_b, c_out, k, stride, h, w), kw = case
    if prec == "tf32" and c_b * 4 % 16:
        pytest.skip("second input below 16 bytes per pixel")
    got, x, p, spec, layer = run_cat(n, c_a, c_b, c_out, k, stride, h, w, prec, B.CBS_NHWC, B.CBS_NHWC, **kw)
    assert layer.plan.variant == PRECS[prec]
    if kw.get("force_window"):
        assert layer.plan.window == 1
    check_tc(prec, got, tc_refs(prec, x, p, spec.stride, spec.pad))


def test_two_input_residual_identity(cuda_lib):
    """Two inputs together with the identity activation and a residual."""
    n, c_a, c_b, c_out, h = 1, 32, 32, 32, 10
    spec = wl.LayerSpec(c_a + c_b, c_out, 3, 1, h)
    x, p = wl.layer_inputs(spec, n, layer_index=22)
    r = np.random.default_rng(9).standard_normal((n, c_out, h, h)).astype(np.float32)
    desc = make_desc(n, c_a + c_b, h, h, c_out, 3, 1, c_in_b=c_b, activation=B.CBS_ACT_IDENTITY, residual=1)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xa = torch.from_numpy(np.ascontiguousarray(x[:, :c_a])).cuda()
    xb = torch.from_numpy(np.ascontiguousarray(x[:, c_a:])).cuda()
    y = layer(xa, residual=torch.from_numpy(r).cuda(), x_b=xb)
    torch.cuda.synchronize()
    want = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1,
                                  act=B.CBS_ACT_IDENTITY, residual=r)
    assert rel_l2(y.cpu().numpy(), want) <= TOL_FP32_REL_L2


@pytest.mark.parametrize("case", [
    ((2, 64, 64, 64, 3, 1, 17, 17), (0, 0)),        # symmetric, 3x3, the junction between channel blocks
    ((1, 96, 32, 48, 3, 2, 21, 19), (-30, 12)),     # asymmetric, stride 2, channel block 32
    ((2, 128, 48, 64, 1, 1, 12, 12), (5, -90)),     # 1x1: 2-D tile boxes, second input padded to 64 codes
])
def test_int8_two_inputs(cuda_lib, case):
    """INT8 two-input layers bit for bit against the oracle on the
    concatenated, quantised input (both inputs share the scale and zero point)."""
    (n, c_a, c_b, c_out, k, stride, h, w), (z_x, z_y) = case
    spec = wl.LayerSpec(c_a + c_b, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=23)
    s_x = float(wl.S_X_INT8)
    y32 = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, stride, spec.pad)
    s_y = float(np.float32(np.abs(y32).max() / 120))
    desc = make_desc(n, c_a + c_b, h, w, c_out, k, stride, spec.pad, prec=B.CBS_INT8, c_in_b=c_b,
                     zero_point_x=z_x, zero_point_y=z_y)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x)
    assert layer.plan.variant == B.CBS_VARIANT_TC_INT8
    xa, xb = layer.pack_inputs(torch.from_numpy(np.ascontiguousarray(x[:, :c_a])).cuda(),
                               torch.from_numpy(np.ascontiguousarray(x[:, c_a:])).cuda())
    y = nhwc_to_nchw(layer(xa, s_y=s_y, x_b=xb).cpu().numpy())
    q_x = oracle.quantize_act(x, s_x, z_x)
    q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x)
    want = oracle.conv_i8(q_x, q_w, bias, m_c, s_y, stride, spec.pad, z_x=z_x, z_y=z_y)
    assert int(np.count_nonzero(y != want)) == 0
