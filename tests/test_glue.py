"""GPU checks of the entry-layout and neck-glue kernels (bit-exact moves)."""
import numpy as np
import pytest
import torch

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc, upsample2x_concat
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


def test_pack_input_fp32_nhwc(cuda_lib):
    spec = wl.LayerSpec(3, 16, 3, 2, 37)
    x, p = wl.layer_inputs(spec, 2)
    desc = make_desc(2, 3, 37, 37, 16, 3, 2, prec=B.CBS_FP32, in_layout=B.CBS_NHWC, out_layout=B.CBS_NHWC)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xp = layer.pack_input(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(xp.cpu().numpy(), x.transpose(0, 2, 3, 1))
