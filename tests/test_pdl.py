"""Programmatic dependent launch changes only when kernels may start: a chain
of dependent layers (each reads the previous layer's output) gives the same
bits with it on and off, eagerly and inside a CUDA graph."""
import numpy as np
import pytest
import torch

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300.chain import Chain

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prec,n,layout", [("bf16", 2, None), ("fp32", 1, None), ("tf32", 1, None),
                                           ("fp32", 1, B.CBS_NHWC)])   # 3xTF32, split-K counters across launches
def test_chain_bits_with_and_without_pdl(cuda_lib, prec, n, layout):
    chain = Chain(prec, n, layout=layout)
    g = torch.Generator().manual_seed(3)
    frame = torch.randn((n, 3, 640, 640), generator=g).cuda()
    outs = {}
    try:
        for opt in (0, B.CBS_LAUNCH_PDL):
            B.cbs_set_launch_options(opt)
            chain.run(frame)
            torch.cuda.synchronize()
            eager = [o.clone() for o in chain.outs]
            for o in chain.outs:
                o.zero_()
            graph = torch.cuda.CUDAGraph()
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(graph, stream=st):
                chain.run(frame, stream=st.cuda_stream)
            for _ in range(2):
                for o in chain.outs:
                    o.zero_()
                torch.cuda.synchronize()
                with torch.cuda.stream(st):
                    graph.replay()
                torch.cuda.synchronize()
                for a, b in zip(eager, chain.outs):
                    assert torch.equal(a, b)
            outs[opt] = eager
    finally:
        B.cbs_set_launch_options(B.CBS_LAUNCH_PDL)
    for a, b in zip(outs[0], outs[B.CBS_LAUNCH_PDL]):
        assert torch.equal(a, b)
    assert all(np.isfinite(o.float().cpu().numpy()).all() for o in outs[0])
