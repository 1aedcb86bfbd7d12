"""A non-finite input reaches exactly the outputs whose windows hold it.

The convolution of page 1 sums the products of each output's k x k window,
so a NaN (or an infinity) in one input pixel makes exactly the outputs of the
windows that contain it non-finite: the oracle's NaN pattern.  Paths that
read more than the window have to keep the extra data out of the sum:
- the stems' pixel-pair K layout carries the pixel left of each window with
  a zero weight, and zero times NaN is NaN, so the kernels zero that pixel;
- windowed A computes the padded grid's extra columns and drops them;
- the tensor cores' channel padding is zero-filled.
Each case plants NaNs and infinities at an interior pixel, at the image edges
and next to the stems' pair boundaries, and compares the non-finite pattern
with the oracle's and the finite values with the precision's bar.
"""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
from helpers import nhwc_to_nchw, rel_l2

pytestmark = pytest.mark.gpu

PRECS = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16}
# Relative L2 bars over the finite outputs (FP32 exact path; TF32/BF16 bar).
BARS = {"fp32": 1e-5, "tf32": 5e-3, "bf16": 5e-3}


def plant(x):
    """NaN and +-inf at fixed pixels: interior, corners, first and last
    columns, and an odd column (the second pixel of a stem pixel pair)."""
    n, c, h, w = x.shape
    x = x.copy()
    spots = [(0, 0, h // 2, w // 2, np.nan), (0, c - 1, 0, 0, np.inf), (n - 1, 0, h - 1, w - 1, -np.inf),
             (n - 1, c // 2, 1, 3, np.nan), (0, 0, h - 2, 5, np.nan), (n - 1, 0, 2, w - 1, np.nan)]
    for (i, ch, r, col, v) in spots:
        x[i, ch, r, col] = v
    return x


@pytest.mark.parametrize("prec,shape,kw", [
    ("bf16", (2, 3, 16, 3, 2, 40, 64), {}),                       # the stem's row kernel (BF16)
    ("tf32", (2, 3, 16, 3, 2, 40, 64), {}),                       # the stem's row kernel (TF32)
    ("bf16", (2, 3, 16, 3, 2, 37, 37), {}),                       # general tensor-core stem, odd width
    ("bf16", (1, 3, 32, 3, 2, 30, 30), {}),                       # general tensor-core stem, pixel pairs
    ("bf16", (2, 64, 64, 3, 1, 12, 12), {"force_window": 1}),     # windowed A
    ("tf32", (2, 32, 48, 3, 2, 14, 14), {}),                      # im2col A, stride 2
    ("fp32", (1, 16, 32, 3, 1, 11, 11), {}),                      # CUDA-core FP32
])
def test_non_finite_inputs_stay_in_their_windows(cuda_lib, prec, shape, kw):
    n, c_in, c_out, k, stride, h, w = shape
    spec = wl.LayerSpec(c_in, c_out, k, stride, h, w)
    x, p = wl.layer_inputs(spec, n, layer_index=6)
    x = plant(x)
    layout = B.CBS_NCHW if prec == "fp32" else B.CBS_NHWC
    d = make_desc(n, c_in, h, w, c_out, k, stride, spec.pad, prec=PRECS[prec], in_layout=layout, **kw)
    layer = FusedConvBnSilu(d, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    xd = torch.from_numpy(x).cuda()
    y = layer(xd if prec == "fp32" else layer.pack_input(xd))
    torch.cuda.synchronize()
    y = y.float().cpu().numpy()
    if layout == B.CBS_NHWC:
        y = nhwc_to_nchw(y)
    else:
        y = y[..., :spec.ow]
    want = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, stride, spec.pad)
    bad_want = ~np.isfinite(want)
    assert bad_want.any() and not bad_want.all()
    assert np.array_equal(~np.isfinite(y), bad_want), (prec, shape, int((~np.isfinite(y) != bad_want).sum()))
    ok = ~bad_want
    assert rel_l2(y[ok], want[ok]) <= BARS[prec], (prec, shape)
