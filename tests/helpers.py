"""Shared helpers for the parity tests (metrics and layout moves on the host)."""
from __future__ import annotations

import numpy as np


def rel_l2(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((got - ref).ravel()) / (den if den > 0 else 1.0))


def max_abs(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64)))) if np.size(ref) else 0.0


def nhwc_to_nchw(a):
    return np.ascontiguousarray(np.asarray(a).transpose(0, 3, 1, 2))


def nchw_to_nhwc(a):
    return np.ascontiguousarray(np.asarray(a).transpose(0, 2, 3, 1))


def max_unit_err(got, ref) -> float:
    """Max abs error on unit-scale outputs: max |got - ref| / max(1, |ref|),
    element by element (an absolute bound where |ref| <= 1, relative above)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if not np.size(ref):
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))


def bf16_round(a) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even) and back to float32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def folded_f32(p):
    """The folded weights and bias as the library's fold computes them: float32
    IEEE operations in the order s = gamma / sqrt(var + eps), w' = w * s,
    b' = beta - mean * s (numpy float32 arithmetic rounds each step to
    nearest, like the fold's explicit round-to-nearest operations)."""
    f = np.float32
    s = (p.gamma.astype(f) / np.sqrt(p.var.astype(f) + f(p.eps))).astype(f)
    w = (p.w.astype(f) * s[:, None, None, None]).astype(f)
    b = (p.beta.astype(f) - (p.mean.astype(f) * s).astype(f)).astype(f)
    return w, b


def bf16_operand_ref(x, p, stride, pad, act=0, residual=None):
    """The oracle evaluated on the operands a BF16 layer multiplies: x and the
    folded weights rounded to bfloat16, the folded bias in float32.  BatchNorm
    is then the identity (gamma 1, mean 0, var 1, eps 0: the oracle divides by
    sqrt(1) = 1 exactly) and beta carries the folded bias."""
    import oracle
    w, b = folded_f32(p)
    c = w.shape[0]
    one, zero = np.ones(c, np.float32), np.zeros(c, np.float32)
    return oracle.conv_bn_act_f32(bf16_round(x), bf16_round(w), one, b, zero, one, 0.0, stride, pad, act=act,
                                  residual=None if residual is None else bf16_round(residual))


def tc_refs(prec, x, p, stride, pad, act=0, residual=None):
    """(oracle on the layer's float32 inputs, reference for the max bound) for
    a TF32 or BF16 layer: the same oracle for TF32, the bfloat16-operand
    oracle for BF16."""
    import oracle
    full = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, stride, pad, act=act,
                                  residual=residual)
    if prec == "bf16":
        return full, bf16_operand_ref(x, p, stride, pad, act=act, residual=residual)
    return full, full


def check_tc(prec, got, refs, what=""):
    """The TF32/BF16 bars: relative L2 <= 5e-3 against the first reference and
    max_unit_err <= 2e-2 against the second (see tc_refs)."""
    e = rel_l2(got, refs[0])
    m = max_unit_err(got, refs[1])
    assert e <= TOL_TC_REL_L2 and m <= TOL_TC_MAX_ABS, (what, e, m)
    return e, m


# FP32 paths: relative L2 <= 1e-5.  TF32/BF16 tensor-core paths: relative
# L2 <= 5e-3 against the oracle on the layer's float32 input, and max abs
# error <= 2e-2 on unit-scale outputs (max_unit_err).  TF32 meets that max
# bound against the same oracle.  BF16 cannot: bfloat16 operands alone (8
# significant bits on x and on the weights) put an exact-arithmetic layer at
# up to 0.033 on the list at batch 16 (tests/test_parity_bar.py measures it),
# so for BF16 the max bound is held against the oracle on the bfloat16
# operands the layer multiplies (bf16_operand_ref).  INT8: exact.
TOL_FP32_REL_L2 = 1e-5
TOL_TC_REL_L2 = 5e-3
TOL_TC_MAX_ABS = 2e-2
