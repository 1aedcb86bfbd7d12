"""The 40-layer chain on INT8 layers, with layers kept in float (page 3,
"Edge optimisation of YOLO26", Highlights: per-channel INT8 weights, and the
layers a sensitivity analysis marks kept in float), against the oracle.

- Seams: cbs_dequantize_i8 and cbs_quantize_i8 bit for bit against the
  oracle's dequantiser (with its bfloat16 rounding) and quantiser.
- Teacher-forced chain (batch 16 all-INT8; batch 4 with layers kept in
  float): the oracle runs the whole chain (INT8 layers on
  codes; layers kept in float on the bfloat16-rounded dequantised input,
  their output rounded to bfloat16 and quantised with the calibrated scale
  for the next INT8 layer).  Each GPU layer is fed the oracle's input for it:
  INT8 layers must return the oracle's codes exactly; layers kept in BF16
  meet the BF16 bars.
- Free-running: the whole chain from the frame, through the library's seams;
  its last output, dequantised, is compared with the FP32 oracle chain and
  the drift is printed (not gated beyond a sanity bound)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.chain import Chain
from conv_bn_silu_gb300.layer import current_stream
from helpers import bf16_operand_ref, check_tc, rel_l2

pytestmark = pytest.mark.gpu

SCALES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "int8_chain_scales.json")))


@pytest.mark.parametrize("count", [16, 1000, 4096 + 7])
@pytest.mark.parametrize("z", [0, -37, 100])
def test_seams_bit_exact(cuda_lib, count, z):
    rng = np.random.default_rng(count * 1000 + z + 500)
    s = np.float32(0.0413)
    q = rng.integers(-128, 128, count).astype(np.int8)
    qd = torch.from_numpy(q).cuda()
    st = current_stream()
    for prec, dt in ((B.CBS_BF16, torch.bfloat16), (B.CBS_FP32, torch.float32)):
        out = torch.empty(count, dtype=dt, device="cuda")
        B.cbs_dequantize_i8(qd, out, count, s, z, prec, st)
        want = oracle.dequantize_i8(q, s, z)
        if dt == torch.bfloat16:
            want = oracle.round_bf16(want)
        assert np.array_equal(out.float().cpu().numpy().view(np.uint32), want.view(np.uint32)), prec
    x = (rng.standard_normal(count) * 3).astype(np.float32)
    x[:8] = np.array([0.5, 1.5, -0.5, -2.5, 1e9, -1e9, 0.0, -0.0], np.float32) * s   # ties, saturation
    for prec, dt in ((B.CBS_BF16, torch.bfloat16), (B.CBS_FP32, torch.float32)):
        xd = torch.from_numpy(x).to(dt).cuda()
        qo = torch.empty(count, dtype=torch.int8, device="cuda")
        B.cbs_quantize_i8(xd, prec, qo, count, s, z, st)
        want = oracle.quantize_act(xd.float().cpu().numpy(), s, z)
        assert np.array_equal(qo.cpu().numpy(), want), prec


def upsample(a):
    return a.repeat(2, axis=2).repeat(2, axis=3)


def oracle_int8_chain(chain, frame):
    """Inputs and outputs of every layer of the chain in the oracle (NCHW):
    int8 codes for INT8 layers, bfloat16-rounded float32 values for layers
    kept in BF16."""
    ins, outs = [], []

    def as_format(j, lp):
        y = outs[j]
        if lp == "int8":
            return y if y.dtype == np.int8 else oracle.quantize_act(y, chain.out_scales[j])
        v = oracle.dequantize_i8(y, chain.out_scales[j]) if y.dtype == np.int8 else y
        return oracle.round_bf16(v)

    for i, cl in enumerate(chain.specs):
        s, src, lp = cl.spec, cl.src, chain.layer_prec[i]
        if src[0] == "frame":
            x = oracle.quantize_act(frame, chain.in_scale) if lp == "int8" else oracle.round_bf16(frame)
        elif src[0] == "layer":
            x = as_format(src[1], lp)
        else:
            x = np.concatenate([upsample(as_format(src[1], lp)), as_format(src[2], lp)], axis=1)
        p = chain.params(i)
        if lp == "int8":
            q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, chain.input_scale(i))
            y = oracle.conv_i8(x, q_w, bias, m_c, chain.out_scales[i], s.stride, s.pad)
        else:
            y = oracle.round_bf16(oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps,
                                                          s.stride, s.pad))
        ins.append(x)
        outs.append(y)
    return ins, outs


def to_device_nhwc(a, dtype, channels):
    """NCHW array -> NHWC device tensor of `dtype` with `channels` channels
    (extra channels zero: code 0 / value 0, as the packing step writes)."""
    t = torch.from_numpy(np.ascontiguousarray(a.transpose(0, 2, 3, 1)))
    t = t.to(torch.int8) if dtype == torch.int8 else t.float().to(dtype)
    if t.shape[-1] < channels:
        t = torch.nn.functional.pad(t.float(), (0, channels - t.shape[-1])).to(dtype)
    return t.contiguous().cuda()


@pytest.mark.parametrize("keep_float,n", [((), 16), ((0, 11, 20, 39), 4)])
def test_int8_chain_teacher_forced(cuda_lib, keep_float, n):
    """All INT8 at batch 16 (every image checked), and with four layers kept
    in BF16 at batch 4."""
    chain = Chain("int8", n, out_scales=SCALES["chain"], keep_float=keep_float)
    assert chain.in_scale == np.float32(SCALES["input_scale"])
    frame = wl.frame(n)
    ins, outs = oracle_int8_chain(chain, frame)
    worst = []
    for i, layer in enumerate(chain.layers):
        lp = chain.layer_prec[i]
        dt = layer.x_dtype
        x = ins[i]
        c_b = layer.desc.c_in_b
        if c_b:
            c_a = x.shape[1] - c_b
            xa = to_device_nhwc(x[:, :c_a], dt, layer.x_shape()[-1])
            xb = to_device_nhwc(x[:, c_a:], dt, layer.x_b_shape()[-1])
        else:
            xa, xb = to_device_nhwc(x, dt, layer.x_shape()[-1]), None
        s_y = chain.out_scales[i] if lp == "int8" else None
        y = layer(xa, s_y=s_y, x_b=xb)
        got = y.float().cpu().numpy().transpose(0, 3, 1, 2) if lp != "int8" else y.cpu().numpy().transpose(0, 3, 1, 2)
        if lp == "int8":
            mism = int(np.count_nonzero(got != outs[i]))
            assert mism == 0, (i, mism, got.size)
        else:
            sp, p = chain.specs[i].spec, chain.params(i)
            full = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, sp.stride, sp.pad)
            e, _ = check_tc("bf16", got, (full, bf16_operand_ref(x, p, sp.stride, sp.pad)), i)
            worst.append(e)
    if worst:
        print(f"kept-in-float layers {keep_float}: worst rel L2 {max(worst):.3e}")

    # Free-running from the frame through the library's seams.
    chain.run(torch.from_numpy(frame).cuda())
    torch.cuda.synchronize()
    last = len(chain.layers) - 1
    y = chain.outs[last]
    if chain.layer_prec[last] == "int8":
        codes = y.cpu().numpy()
        assert len(np.unique(codes)) > 20
        yv = oracle.dequantize_i8(codes, chain.out_scales[last])
    else:
        yv = y.float().cpu().numpy()
    # The FP32 oracle chain's last output, for the drift.
    ref = frame
    fouts = []
    for i, cl in enumerate(chain.specs):
        s, src = cl.spec, cl.src
        xin = ref if src[0] == "frame" else fouts[src[1]] if src[0] == "layer" else \
            np.concatenate([upsample(fouts[src[1]]), fouts[src[2]]], axis=1)
        p = chain.params(i)
        fouts.append(oracle.conv_bn_silu_f32(xin, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad))
    drift = rel_l2(yv.transpose(0, 3, 1, 2), fouts[last])
    print(f"INT8 chain keep_float={keep_float}: last layer vs the FP32 oracle chain, rel L2 {drift:.3e}")
    assert np.isfinite(yv).all() and drift < 1.0
