"""GPU checks of the entry-layout and neck-glue kernels (bit-exact moves)."""
import numpy as np
import pytest
import torch

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc, upsample2x, upsample2x_concat
from conv_bn_silu_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _np_upcat_nhwc(a, b):
    up = a.repeat(2, axis=1).repeat(2, axis=2)
    return np.concatenate([up, b], axis=3)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int8])
@pytest.mark.parametrize("ca,cb", [(256, 128), (3, 5), (8, 8)])
def test_upsample_concat_nhwc(cuda_lib, dtype, ca, cb):
    g = torch.Generator().manual_seed(ca * 7 + cb)
    a = (torch.randn((2, 5, 6, ca), generator=g, dtype=torch.float32) * 50).to(dtype)
    b = (torch.randn((2, 10, 12, cb), generator=g, dtype=torch.float32) * 50).to(dtype)
    out = upsample2x_concat(a.cuda(), b.cuda(), B.CBS_NHWC)
    torch.cuda.synchronize()
    ref = _np_upcat_nhwc(a.view(torch.int8 if dtype == torch.int8 else torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy(),
                         b.view(torch.int8 if dtype == torch.int8 else torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy())
    got = out.cpu().view(torch.int8 if dtype == torch.int8 else torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy()
    assert np.array_equal(got, ref)


def test_upsample_concat_nchw(cuda_lib):
    g = torch.Generator().manual_seed(3)
    a = torch.randn((2, 7, 4, 5), generator=g, dtype=torch.float32)
    b = torch.randn((2, 3, 8, 10), generator=g, dtype=torch.float32)
    out = upsample2x_concat(a.cuda(), b.cuda(), B.CBS_NCHW).cpu()
    ref = torch.cat([a.repeat_interleave(2, 2).repeat_interleave(2, 3), b], 1)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_upsample_only(cuda_lib, layout, dtype):
    """cb = 0: the plain upsample that feeds a two-input layer."""
    g = torch.Generator().manual_seed(11)
    shape = (2, 5, 6, 24) if layout == B.CBS_NHWC else (2, 24, 5, 6)
    a = (torch.randn(shape, generator=g) * 10).to(dtype)
    out = upsample2x(a.cuda(), layout).cpu()
    hw = (1, 2) if layout == B.CBS_NHWC else (2, 3)
    assert torch.equal(out, a.repeat_interleave(2, hw[0]).repeat_interleave(2, hw[1]))


def test_pack_input_fp32_nhwc(cuda_lib):
    spec = wl.LayerSpec(3, 16, 3, 2, 37)
    x, p = wl.layer_inputs(spec, 2)
    desc = make_desc(2, 3, 37, 37, 16, 3, 2, prec=B.CBS_FP32, in_layout=B.CBS_NHWC, out_layout=B.CBS_NHWC)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xp = layer.pack_input(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(xp.cpu().numpy(), x.transpose(0, 2, 3, 1))


@pytest.mark.parametrize("prec", [B.CBS_BF16, B.CBS_INT8, B.CBS_TF32])
@pytest.mark.parametrize("c_in", [3, 8, 24])
@pytest.mark.parametrize("w", [21, 24])
def test_pack_input_nhwc_exact(cuda_lib, prec, c_in, w):
    """Entry packing to NHWC, padded channels zero: bf16 round-to-nearest-even,
    int8 q = rne(clamp(x / s_x, -128, 127)), float copied; few channels take
    the one-thread-per-pixel kernel (four pixels per thread when 4 padded
    channels and W a multiple of 4), more the tiled transpose."""
    n, h = 2, 19
    spec = wl.LayerSpec(c_in, 32, 3, 1, h, w)
    x, p = wl.layer_inputs(spec, n)
    s_x = 0.0125
    desc = make_desc(n, c_in, h, w, 32, 3, 1, prec=prec, in_layout=B.CBS_NHWC, out_layout=B.CBS_NHWC)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x)
    got = layer.pack_input(torch.from_numpy(x).cuda()).cpu()
    c_pad = layer.plan.c_in_pad
    xt = torch.zeros((n, h, w, c_pad), dtype=torch.float32)
    xt[..., :c_in] = torch.from_numpy(x).permute(0, 2, 3, 1)
    if prec == B.CBS_BF16:
        assert torch.equal(got.view(torch.int16), xt.to(torch.bfloat16).view(torch.int16))
    elif prec == B.CBS_INT8:
        q = np.rint(np.clip(xt.numpy() / np.float32(s_x), -128, 127)).astype(np.int8)
        assert np.array_equal(got.numpy(), q)
    else:
        assert torch.equal(got, xt)


def _pool_ref(x_nchw_f32, k, stride, pad):
    import oracle
    return oracle.maxpool2d_f32(x_nchw_f32, k, stride, pad)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int8])
@pytest.mark.parametrize("layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("k,stride,pad,hw,c", [(5, 1, 2, (20, 20), 128), (3, 2, 1, (17, 13), 24), (2, 2, 0, (9, 11), 7),
                                               (5, 1, 2, (1, 3), 16)])
def test_maxpool(cuda_lib, dtype, layout, k, stride, pad, hw, c):
    """Max pooling against the oracle, bit for bit (a max is exact)."""
    from conv_bn_silu_gb300.layer import maxpool2d
    g = torch.Generator().manual_seed(k * 100 + c)
    x = torch.randn((2, c) + hw, generator=g) * 30
    x = x.to(dtype) if dtype != torch.int8 else x.round().clamp(-128, 127).to(torch.int8)
    want = _pool_ref(x.float().numpy(), k, stride, pad)
    xd = x.cuda() if layout == B.CBS_NCHW else x.permute(0, 2, 3, 1).contiguous().cuda()
    y = maxpool2d(xd, k, stride, pad, layout).cpu()
    if layout == B.CBS_NHWC:
        y = y.permute(0, 3, 1, 2)
    assert np.array_equal(y.float().numpy(), want)


def test_maxpool_sppf_chain_and_nan(cuda_lib):
    """SPPF's three 5x5 stride-1 pools in sequence (NHWC bf16), and NaN
    propagation (float)."""
    from conv_bn_silu_gb300.layer import maxpool2d
    g = torch.Generator().manual_seed(5)
    x = torch.randn((2, 256, 20, 20), generator=g).to(torch.bfloat16)
    xd = x.permute(0, 2, 3, 1).contiguous().cuda()
    ref = x.float().numpy()
    for _ in range(3):
        xd = maxpool2d(xd, 5, 1, 2, B.CBS_NHWC)
        ref = _pool_ref(ref, 5, 1, 2)
    assert np.array_equal(xd.permute(0, 3, 1, 2).float().cpu().numpy(), ref)
    xf = torch.randn((1, 3, 6, 6), generator=g)
    xf[0, 1, 2, 2] = float("nan")
    y = maxpool2d(xf.cuda(), 3, 1, 1, B.CBS_NCHW).cpu().numpy()
    want = _pool_ref(xf.numpy(), 3, 1, 1)
    assert np.array_equal(np.isnan(y), np.isnan(want)) and np.array_equal(y[~np.isnan(y)], want[~np.isnan(want)])
