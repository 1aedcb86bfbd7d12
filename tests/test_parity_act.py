"""GPU parity of the identity-activation and residual-add epilogues
(y = act(BN(conv(x))) + r) against the CPU oracle, in every float variant:
the CUDA-core implicit GEMM (with split-K and padded NCHW rows), the direct
small-channel kernel, and the TF32/BF16 tensor-core kernel (staged NHWC
stores, direct stores, windowed A).  Bars as for the fused layer."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import TOL_FP32_REL_L2, bf16_round, check_tc, nchw_to_nhwc, nhwc_to_nchw, rel_l2, tc_refs

pytestmark = pytest.mark.gpu

PRECS = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16}


def run(spec, n, prec, act, with_res, in_layout, out_layout, in_place=False, **kw):
    x, p = wl.layer_inputs(spec, n, layer_index=15)
    r = np.random.default_rng(5).standard_normal((n, spec.c_out, spec.oh, spec.ow)).astype(np.float32)
    if prec == "bf16":
        r = bf16_round(r)
    desc = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad, prec=PRECS[prec],
                     in_layout=in_layout, out_layout=out_layout, activation=act, residual=int(with_res), **kw)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xd = torch.from_numpy(x).cuda()
    xin = xd if (prec == "fp32" and in_layout == B.CBS_NCHW) else layer.pack_input(xd)
    y = layer.empty_y()
    res_dev = None
    if with_res:
        rr = r if out_layout == B.CBS_NCHW else nchw_to_nhwc(r)
        res_dev = torch.from_numpy(np.ascontiguousarray(rr)).to(y.dtype).cuda()
        if out_layout == B.CBS_NCHW and layer.plan.out_row_stride != spec.ow:
            pad = torch.zeros(y.shape, dtype=y.dtype, device="cuda")
            pad[..., :spec.ow] = res_dev
            res_dev = pad
        if in_place:
            y.copy_(res_dev)
            res_dev = y
    layer(xin, y, residual=res_dev)
    torch.cuda.synchronize()
    out = y.float().cpu().numpy()
    if out_layout == B.CBS_NHWC:
        out = nhwc_to_nchw(out)
    out = out[..., :spec.ow]
    if prec == "fp32":
        ref = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad,
                                     act=act, residual=r if with_res else None)
        refs = (ref, ref)
    else:
        refs = tc_refs(prec, x, p, spec.stride, spec.pad, act=act, residual=r if with_res else None)
    return out, refs[0], refs[1], layer


def check(prec, out, ref_x, ref_max, what):
    if prec == "fp32":
        e = rel_l2(out, ref_x)
        assert e <= TOL_FP32_REL_L2, (what, e)
    else:
        check_tc(prec, out, (ref_x, ref_max), what)


@pytest.mark.parametrize("act,with_res", [(B.CBS_ACT_IDENTITY, False), (B.CBS_ACT_SILU, True),
                                          (B.CBS_ACT_IDENTITY, True)])
@pytest.mark.parametrize("layouts", [(B.CBS_NCHW, B.CBS_NCHW), (B.CBS_NHWC, B.CBS_NHWC)])
@pytest.mark.parametrize("split", [1, 3])
def test_cuda_core(cuda_lib, act, with_res, layouts, split):
    spec = wl.LayerSpec(24, 40, 3, 1, 17)
    out, rx, rr, layer = run(spec, 2, "fp32", act, with_res, *layouts, force_variant=B.CBS_VARIANT_SIMT_FP32,
                             force_split_k=split)
    assert layer.plan.split_k == split
    check("fp32", out, rx, rr, (act, with_res, layouts, split))


def test_cuda_core_padded_rows_in_place(cuda_lib):
    """NCHW rows with a padded pitch; the residual is y itself."""
    spec = wl.LayerSpec(16, 32, 3, 1, 20)
    out, rx, rr, _ = run(spec, 1, "fp32", B.CBS_ACT_IDENTITY, True, B.CBS_NCHW, B.CBS_NCHW, in_place=True,
                         out_row_stride=32)
    check("fp32", out, rx, rr, "padded in place")


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
@pytest.mark.parametrize("act,with_res", [(B.CBS_ACT_IDENTITY, False), (B.CBS_ACT_SILU, True),
                                          (B.CBS_ACT_IDENTITY, True)])
@pytest.mark.parametrize("out_layout", [B.CBS_NCHW, B.CBS_NHWC])
def test_small_channel_kernel(cuda_lib, prec, act, with_res, out_layout):
    spec = wl.LayerSpec(3, 16, 3, 2, 26)
    in_layout = B.CBS_NCHW if prec == "fp32" else B.CBS_NHWC
    out, rx, rr, layer = run(spec, 2, prec, act, with_res, in_layout, out_layout)
    assert layer.plan.variant == B.CBS_VARIANT_STEM
    check(prec, out, rx, rr, (prec, act, with_res, out_layout))


TC_CASES = [
    # (spec, n, out_layout, extra descriptor fields)
    (wl.LayerSpec(64, 64, 3, 1, 12), 2, B.CBS_NHWC, {}),                       # staged TMA stores
    (wl.LayerSpec(32, 48, 3, 2, 15), 2, B.CBS_NCHW, {}),                       # direct NCHW stores
    (wl.LayerSpec(16, 20, 1, 1, 9), 3, B.CBS_NHWC, {}),                        # BF16 rows of 40 B: direct stores
    (wl.LayerSpec(64, 96, 3, 1, 10), 2, B.CBS_NHWC, {"force_window": 1}),      # windowed A
    (wl.LayerSpec(64, 272, 1, 1, 8), 2, B.CBS_NHWC, {"force_block_m": 256}),   # two sub-tiles, several N tiles
]


@pytest.mark.parametrize("prec", ["bf16", "tf32"])
@pytest.mark.parametrize("act,with_res", [(B.CBS_ACT_IDENTITY, False), (B.CBS_ACT_SILU, True),
                                          (B.CBS_ACT_IDENTITY, True)])
@pytest.mark.parametrize("case", range(len(TC_CASES)))
def test_tensor_cores(cuda_lib, prec, act, with_res, case):
    spec, n, out_layout, kw = TC_CASES[case]
    out, rx, rr, layer = run(spec, n, prec, act, with_res, B.CBS_NHWC, out_layout, **kw)
    assert layer.plan.variant in (B.CBS_VARIANT_TC_TF32, B.CBS_VARIANT_TC_BF16)
    check(prec, out, rx, rr, (prec, act, with_res, case))


def test_no_timeout_reported(cuda_lib):
    assert B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream) == B.CBS_OK
