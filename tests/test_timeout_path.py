"""The timeout path of the bounded device waits, exercised without a fault.

Every mbarrier wait in the tensor-core kernels gives up after a time limit,
records CBS_ERR_TIMEOUT in the library's status word and lets the kernel
return.  cbs_selftest_wait_timeout runs that same bounded wait on a barrier
nothing arrives at, with a limit of a few milliseconds; the test checks that
cbs_read_device_status reports the timeout, that a reset clears it, and that
the context still runs a layer correctly afterwards."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.layer import FusedConvBnSilu, current_stream, make_desc
from helpers import TOL_FP32_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_is_reported(cuda_lib):
    s = current_stream()
    assert B.cbs_read_device_status(True, s) == B.CBS_OK
    B.cbs_selftest_wait_timeout(3000, s)
    assert B.cbs_read_device_status(False, s) == B.CBS_ERR_TIMEOUT
    assert B.cbs_read_device_status(True, s) == B.CBS_ERR_TIMEOUT     # read, then cleared
    assert B.cbs_read_device_status(False, s) == B.CBS_OK
    # The context is still usable: a tensor-core layer runs and matches the oracle.
    spec = wl.LayerSpec(16, 32, 3, 1, 12)
    x, p = wl.layer_inputs(spec, 2, layer_index=3)
    desc = make_desc(2, 16, 12, 12, 32, 3, 1, prec=B.CBS_FP32, in_layout=B.CBS_NHWC, out_layout=B.CBS_NCHW)
    layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
    y = layer(layer.pack_input(torch.from_numpy(x).cuda())).cpu().numpy()
    want = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1)
    assert rel_l2(y, want) <= TOL_FP32_REL_L2
    assert B.cbs_read_device_status(True, s) == B.CBS_OK


def test_selftest_rejects_limits_out_of_range(cuda_lib):
    for bad in (0, -5, 100001):
        with pytest.raises(B.CbsError) as e:
            B.cbs_selftest_wait_timeout(bad, None)
        assert e.value.status == B.CBS_ERR_INVALID_ARG
