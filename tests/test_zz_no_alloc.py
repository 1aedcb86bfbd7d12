"""The allocation-free entry point (cbs_conv_bn_silu_f32_noalloc).

Callers such as plugin interfaces that pass only input and output pointers,
or serving loops that must not allocate after start-up, cannot provide the
split-K workspace the regular entry point takes.  This entry point uses the
library's own fixed device array instead.  The test runs a split-K layer
through it twice in a row (the second call finds the first call's scratch
contents) and compares each result with the regular entry point's: the two run the
same kernel and sum the split-K parts in the same fixed order, so the
results must be identical bit for bit (anything else means the scratch was
corrupted).  Each result is also held to the FP32 bar against the oracle.  It passes alone in a fresh process and after the
other tests; the file name makes pytest collect it last."""
import numpy as np
import pytest
import torch

import oracle

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, current_stream, make_desc
from helpers import TOL_FP32_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("split", [6, 16])
def test_noalloc_matches_regular_entry_point_twice(cuda_lib, split):
    spec = wl.LayerSpec(256, 256, 3, 1, 20)
    x, p = wl.layer_inputs(spec, 1, layer_index=10)
    desc = make_desc(1, 256, 20, 20, 256, 3, 1, force_split_k=split)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    assert layer.plan.split_k == split and layer.plan.workspace_bytes > 0
    xd = torch.from_numpy(x).cuda()
    ref = layer(xd).cpu().numpy()                      # regular entry point, caller workspace
    want = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1)
    for _ in range(2):
        y = torch.full(layer.y_shape(), float("nan"), dtype=torch.float32, device="cuda")
        B.cbs_conv_bn_silu_f32_noalloc(layer.plan, xd, layer.w_packed, layer.bias, y, current_stream())
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.array_equal(got, ref)
        assert rel_l2(got, want) <= TOL_FP32_REL_L2


def test_noalloc_rejects_oversized_plan(cuda_lib):
    # 1x1 conv over a large batch with a forced split: scratch above 16 MiB.
    desc = make_desc(16, 256, 80, 80, 256, 1, 1, force_split_k=8)
    plan = B.cbs_plan(desc)
    assert plan.workspace_bytes > 16 << 20
    with pytest.raises(B.CbsError) as e:
        B.cbs_conv_bn_silu_f32_noalloc(plan, 1 << 20, 1 << 20, 1 << 20, 1 << 20, current_stream())
    assert e.value.status == B.CBS_ERR_WORKSPACE
