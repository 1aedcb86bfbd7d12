"""The 40-layer whole-frame chain on the GPU against the CPU oracle.

Pass/fail is teacher-forced: every GPU layer is fed the oracle's input for
that layer (packed into the layer's format by cbs_pack_input) and its output
is compared with the oracle's, with the bars of its variant (FP32: relative
L2 <= 1e-5; TF32/BF16: relative L2 <= 5e-3 and max |err| / max(1, |ref|)
<= 2e-2, for BF16 against the oracle on the bfloat16 operands).  The
free-running chain (each GPU layer on the GPU output before it) is checked
for finiteness and its drift is printed.

FP32 runs at batch 1 (the frame config); TF32 and BF16 at batch 16, the
throughput config, with all 16 images checked."""
import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.chain import Chain, to_nchw_numpy
from helpers import TOL_FP32_REL_L2, bf16_operand_ref, check_tc, rel_l2

pytestmark = pytest.mark.gpu


def upcat(a, b):
    """Neck glue on NCHW arrays: concat(upsample2x(a), b) along channels."""
    return np.concatenate([a.repeat(2, axis=2).repeat(2, axis=3), b], axis=1)


def sppf_cat(a):
    """SPPF glue on an NCHW array: concat(a, p(a), p(p(a)), p(p(p(a)))), p the
    5x5 stride-1 max pool with padding 2 (the oracle's pool applied three times)."""
    parts, cur = [a], a
    for _ in range(3):
        cur = oracle.maxpool2d_f32(cur, wl.SPPF_POOL_K, 1, wl.SPPF_POOL_K // 2)
        parts.append(cur)
    return np.concatenate(parts, axis=1)


def oracle_chain(chain, frame):
    """Oracle inputs and outputs of every layer (NCHW float32)."""
    ins, outs = [], []
    for i, cl in enumerate(chain.specs):
        s, src = cl.spec, cl.src
        if src[0] == "frame":
            x = frame
        elif src[0] == "layer":
            x = outs[src[1]]
        elif src[0] == "sppf":
            x = sppf_cat(outs[src[1]])
        else:
            x = upcat(outs[src[1]], outs[src[2]])
        p = chain.params(i)
        ins.append(x)
        outs.append(oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad))
    return ins, outs


@pytest.mark.parametrize("prec,n,layout,sppf", [("fp32", 1, None, False), ("fp32", 1, B.CBS_NHWC, False),
                                                ("tf32", 16, None, False), ("bf16", 16, None, False),
                                                ("fp32", 1, None, True), ("bf16", 16, None, True)])
def test_chain_teacher_forced(cuda_lib, prec, n, layout, sppf):
    """FP32 in NHWC runs the 3xTF32 tensor-core variant (split-K on the small
    layers) and is held to the FP32 bar like the CUDA-core chain.  With sppf,
    the whole synthetic frame: the SPPF block (1x1 conv, the three chained
    pools in one glue kernel, 1x1 conv over the four-way concatenation read
    as two inputs) after layer 10; its free-running run also checks the pool
    glue inside the frame."""
    chain = Chain(prec, n, layout=layout, sppf=sppf)
    frame = wl.frame(n)
    ins, outs = oracle_chain(chain, frame)
    s = torch.cuda.current_stream().cuda_stream
    worst = []
    for i, layer in enumerate(chain.layers):
        x_full = ins[i]
        c_b = layer.desc.c_in_b
        if c_b:   # two-input layer: its inputs are the two parts of the concatenation
            c_a = x_full.shape[1] - c_b
            xa, xb = layer.pack_inputs(torch.from_numpy(np.ascontiguousarray(x_full[:, :c_a])).cuda(),
                                       torch.from_numpy(np.ascontiguousarray(x_full[:, c_a:])).cuda())
            got = to_nchw_numpy(layer(xa, x_b=xb), chain.layout)
        else:
            xin = layer.empty_x()
            B.cbs_pack_input(layer.plan, torch.from_numpy(x_full).cuda(), xin, 0.0, s)
            got = to_nchw_numpy(layer(xin), chain.layout)
        assert got.shape == outs[i].shape
        if prec == "fp32":
            e = rel_l2(got, outs[i])
            assert e <= TOL_FP32_REL_L2, (i, e)
        else:
            sp = chain.specs[i].spec
            ref_max = outs[i] if prec == "tf32" else bf16_operand_ref(x_full, chain.params(i), sp.stride, sp.pad)
            e, _ = check_tc(prec, got, (outs[i], ref_max), i)
        worst.append(e)
    print(f"{prec} n={n} sppf={sppf}: teacher-forced worst rel L2 {max(worst):.3e}")

    # Free-running chain from the frame.
    frame_dev = torch.from_numpy(frame).cuda()
    chain.run(frame_dev)
    torch.cuda.synchronize()
    drift = []
    for i in range(len(chain.layers)):
        y = to_nchw_numpy(chain.outs[i], chain.layout)
        assert np.isfinite(y).all(), i
        drift.append(rel_l2(y, outs[i]))
    print(f"{prec} n={n} sppf={sppf}: free-running drift, last layer {drift[-1]:.3e}, max {max(drift):.3e}")
    assert max(drift) < 0.2
