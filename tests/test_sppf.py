"""The SPPF glue (cbs_sppf_pool) against the oracle: three chained k x k
stride-1 max pools with padding k/2, written side by side along channels,
bit for bit equal to applying the oracle's max pool three times (float,
bfloat16 and int8 codes; NHWC and NCHW; ragged tiles and channel groups; a
NaN spreading through the windows)."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300.layer import sppf_pool

pytestmark = pytest.mark.gpu

DT = {"fp32": torch.float32, "bf16": torch.bfloat16, "int8": torch.int8}


def oracle_sppf(x, k):
    """concat(p(x), p(p(x)), p(p(p(x)))) on an NCHW float32 array."""
    outs, cur = [], x
    for _ in range(3):
        cur = oracle.maxpool2d_f32(cur, k, 1, k // 2)
        outs.append(cur)
    return np.concatenate(outs, axis=1)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "int8"])
@pytest.mark.parametrize("layout", [B.CBS_NHWC, B.CBS_NCHW])
@pytest.mark.parametrize("shape", [
    (2, 128, 20, 20, 5),     # the frame's SPPF at 20x20
    (1, 24, 37, 29, 5),      # ragged 16x16 tiles; channels not a multiple of the channel group
    (3, 40, 7, 5, 3),        # 3x3 pools, image smaller than a tile
    (1, 16, 33, 18, 7),      # 7x7 pools
    (2, 8, 1, 1, 5),         # a 1x1 image: every pool returns its input
])
def test_sppf_pool_matches_three_oracle_pools(cuda_lib, dtype, layout, shape):
    n, c, h, w, k = shape
    rng = np.random.default_rng(hash(shape) % 2**32)
    if dtype == "int8":
        x = rng.integers(-128, 128, size=(n, c, h, w)).astype(np.float32)
    else:
        x = rng.standard_normal((n, c, h, w)).astype(np.float32)
        if dtype == "bf16":
            x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    want = oracle_sppf(x, k)
    t = torch.from_numpy(x).to(DT[dtype])
    if layout == B.CBS_NHWC:
        t = t.permute(0, 2, 3, 1)
    got = sppf_pool(t.contiguous().cuda(), k, layout)
    torch.cuda.synchronize()
    got = got.float().cpu().numpy()
    if layout == B.CBS_NHWC:
        got = got.transpose(0, 3, 1, 2)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_sppf_pool_nan_spreads(cuda_lib, dtype):
    x = np.random.default_rng(3).standard_normal((1, 8, 23, 21)).astype(np.float32)
    x[0, 3, 11, 10] = np.nan
    want = oracle_sppf(x, 5)
    got = sppf_pool(torch.from_numpy(x).to(DT[dtype]).permute(0, 2, 3, 1).contiguous().cuda(), 5, B.CBS_NHWC)
    got = got.float().cpu().numpy().transpose(0, 3, 1, 2)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.isnan(want).sum() == 25 + 81 + 169
    ok = ~np.isnan(want)
    wr = want if dtype == "fp32" else torch.from_numpy(want).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got[ok], wr[ok])


def test_sppf_pool_rejects_bad_shapes(cuda_lib):
    for k in (4, 9, 0):
        with pytest.raises(B.CbsError) as e:
            B.cbs_sppf_pool(1 << 20, 1 << 20, 1, 8, 10, 10, k, B.CBS_NHWC, B.CBS_FP32, None)
        assert e.value.status == B.CBS_ERR_INVALID_ARG
