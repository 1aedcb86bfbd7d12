"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test fixes a part of the oracle with something independent of it: a
matrix product, delta kernels, a closed-form count of the zero-padded taps,
BatchNorm identities and PyTorch's own float64 routines, the analytic SiLU
minimum, brute-force im2col on 4x4 inputs, exp against float64, round-half-
even ties, and exact integer sums.  A dropped term, a wrong sign, a
transposed operand or a wrong index in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conv_bn_silu_gb300 import workloads as wl


def rng(seed=0):
    return np.random.default_rng(seed)


def f32(a):
    return np.asarray(a, dtype=np.float32)


def torch_layer(x, w, gamma, beta, mean, var, eps, stride, pad):
    """PyTorch CPU float64 conv2d -> batch_norm -> silu (an independent library)."""
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))  # noqa: E731
    z = torch.nn.functional.conv2d(t(x), t(w), stride=stride, padding=pad)
    b = torch.nn.functional.batch_norm(z, t(mean), t(var), t(gamma), t(beta), training=False,
                                       eps=float(np.float32(eps)))
    return torch.nn.functional.silu(b).numpy(), z.numpy()


# ------------------------------------------------------------------ convolution
def test_conv1x1_is_matrix_product():
    r = rng(1)
    x = f32(r.standard_normal((2, 5, 3, 4)))
    w = f32(r.standard_normal((6, 5, 1, 1)))
    z = oracle.conv2d(x, w, stride=1, pad=0)
    ref = np.einsum("oc,nchw->nohw", w[:, :, 0, 0].astype(np.float64), x.astype(np.float64))
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-13)


def test_delta_kernel_is_identity():
    r = rng(2)
    x = f32(r.standard_normal((2, 4, 5, 7)))
    w = np.zeros((4, 4, 3, 3), np.float32)
    for c in range(4):
        w[c, c, 1, 1] = 1.0
    z = oracle.conv2d(x, w, stride=1, pad=1)
    assert np.array_equal(z, x.astype(np.float64))


def test_shifted_delta_shifts_with_zero_fill():
    r = rng(3)
    x = f32(r.standard_normal((1, 2, 5, 6)))
    w = np.zeros((2, 2, 3, 3), np.float32)
    w[0, 1, 0, 2] = 1.0   # out channel 0 reads in channel 1 at tap (r=0, s=2)
    w[1, 0, 2, 0] = 1.0   # out channel 1 reads in channel 0 at tap (r=2, s=0)
    z = oracle.conv2d(x, w, stride=1, pad=1)
    exp = np.zeros_like(z)
    H, W = 5, 6
    for oh in range(H):
        for ow in range(W):
            ih, iw = oh - 1, ow + 1
            if 0 <= ih < H and 0 <= iw < W:
                exp[0, 0, oh, ow] = x[0, 1, ih, iw]
            ih, iw = oh + 1, ow - 1
            if 0 <= ih < H and 0 <= iw < W:
                exp[0, 1, oh, ow] = x[0, 0, ih, iw]
    assert np.array_equal(z, exp)


@pytest.mark.parametrize("stride", [1, 2])
@pytest.mark.parametrize("hw", [(5, 5), (4, 7)])
def test_zero_padding_closed_form(stride, hw):
    """All-ones input and weights: each output counts its in-image taps
    (4 at corners, 6 on edges, 9 inside for 3x3, times C_in)."""
    H, W = hw
    C_in, k, pad = 3, 3, 1
    x = np.ones((1, C_in, H, W), np.float32)
    w = np.ones((2, C_in, k, k), np.float32)
    z = oracle.conv2d(x, w, stride=stride, pad=pad)
    OH, OW = (H + 2 * pad - k) // stride + 1, (W + 2 * pad - k) // stride + 1
    assert z.shape == (1, 2, OH, OW)
    for oh in range(OH):
        rows = len(set(range(oh * stride - pad, oh * stride - pad + k)) & set(range(H)))
        for ow in range(OW):
            cols = len(set(range(ow * stride - pad, ow * stride - pad + k)) & set(range(W)))
            assert z[0, 0, oh, ow] == C_in * rows * cols == z[0, 1, oh, ow]
    if stride == 1 and hw == (5, 5):
        assert z[0, 0, 0, 0] == 12 and z[0, 0, 0, 2] == 18 and z[0, 0, 2, 2] == 27


def _im2col_conv(x, w, stride, pad):
    """Brute-force reference: explicit im2col matrix times the weight matrix."""
    N, C, H, W = x.shape
    O, _, k, _ = w.shape
    OH, OW = (H + 2 * pad - k) // stride + 1, (W + 2 * pad - k) // stride + 1
    cols = np.zeros((N * OH * OW, C * k * k))
    for n in range(N):
        for oh in range(OH):
            for ow in range(OW):
                row = (n * OH + oh) * OW + ow
                for c in range(C):
                    for r in range(k):
                        for s in range(k):
                            ih, iw = oh * stride - pad + r, ow * stride - pad + s
                            if 0 <= ih < H and 0 <= iw < W:
                                cols[row, (c * k + r) * k + s] = x[n, c, ih, iw]
    out = cols @ w.reshape(O, -1).astype(np.float64).T
    return out.reshape(N, OH, OW, O).transpose(0, 3, 1, 2)


@pytest.mark.parametrize("k,stride,pad", [(1, 1, 0), (1, 2, 0), (3, 1, 0), (3, 1, 1), (3, 2, 0), (3, 2, 1)])
@pytest.mark.parametrize("c_in,c_out", [(1, 1), (2, 3), (3, 2)])
def test_brute_force_4x4(k, stride, pad, c_in, c_out):
    r = rng(10 + k * 7 + stride * 3 + pad + c_in * 11 + c_out)
    x = f32(r.standard_normal((2, c_in, 4, 4)))
    w = f32(r.standard_normal((c_out, c_in, k, k)))
    z = oracle.conv2d(x, w, stride=stride, pad=pad)
    np.testing.assert_allclose(z, _im2col_conv(x, w, stride, pad), rtol=1e-13, atol=1e-13)


# -------------------------------------------------------------------- BatchNorm
def test_bn_identity():
    eps = 2.0 ** -10
    r = rng(4)
    t = r.standard_normal((2, 3, 4, 5))
    C = 3
    out = oracle.batchnorm(t, np.ones(C), np.zeros(C), np.zeros(C), np.full(C, 1 - eps), eps)
    assert np.array_equal(out, t)


def test_bn_matches_torch():
    r = rng(5)
    t = r.standard_normal((2, 6, 4, 4))
    g, b, m = f32(r.uniform(0.5, 1.5, 6)), f32(r.normal(0, 0.3, 6)), f32(r.normal(0, 0.3, 6))
    v = f32(r.uniform(0.5, 2.0, 6))
    out = oracle.batchnorm(t, g, b, m, v, 1e-3)
    ref = torch.nn.functional.batch_norm(torch.from_numpy(t.astype(np.float64)),
                                         *(torch.from_numpy(a.astype(np.float64)) for a in (m, v, g, b)),
                                         training=False, eps=float(np.float32(1e-3))).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_bn_folded_equals_unfused_exact():
    """gamma=2, var+eps=1 makes the fold exact in float32: conv with w*2 and
    bias beta-2*mean must reproduce BN(conv) to rounding of double sums."""
    eps = 2.0 ** -10
    r = rng(6)
    x = f32(r.standard_normal((1, 4, 6, 6)))
    w = f32(r.standard_normal((5, 4, 3, 3)))
    gamma = np.full(5, 2.0, np.float32)
    beta = f32(np.round(r.normal(0, 1, 5) * 64) / 64)
    mean = f32(np.round(r.normal(0, 1, 5) * 64) / 64)
    var = np.full(5, 1.0 - eps, np.float32)
    unfused = oracle.batchnorm(oracle.conv2d(x, w, 1, 1), gamma, beta, mean, var, eps)
    folded = oracle.conv2d(x, w * 2.0, 1, 1, conv_bias=beta - 2.0 * mean)
    np.testing.assert_allclose(folded, unfused, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------ SiLU
def test_silu_special_values():
    xs = np.array([0.0, 1.0, -1.0, 3.5, -3.5, 40.0, -40.0, 800.0, -800.0])
    y = oracle.silu(xs)
    assert y[0] == 0.0
    np.testing.assert_allclose(y[1] - y[2], 1.0, rtol=0, atol=4e-16)    # SiLU(x)-SiLU(-x)=x
    np.testing.assert_allclose(y[3] - y[4], 3.5, rtol=0, atol=4e-15)
    assert abs(y[5] / 40.0 - 1.0) < 1e-15                               # SiLU(x)/x -> 1
    assert -1e-15 < y[6] < 0.0                                          # SiLU(x) -> 0-
    assert y[7] == 800.0 and y[8] == 0.0 and math.copysign(1.0, y[8]) < 0   # e^800 overflows: -0


def test_silu_minimum():
    """The minimum solves 1 + x(1 - sigma(x)) = 0, where SiLU(x) = x + 1."""
    from scipy.optimize import brentq
    xmin = brentq(lambda x: 1 + x * (1 - 1 / (1 + math.exp(-x))), -2.0, -1.0, xtol=1e-15)
    grid = np.linspace(xmin - 1e-3, xmin + 1e-3, 20001)
    y = oracle.silu(grid)
    i = int(np.argmin(y))
    assert abs(grid[i] - xmin) < 2e-7
    assert abs(y[i] - (xmin + 1.0)) < 1e-12
    assert abs(xmin - (-1.2784645427610738)) < 1e-12


# --------------------------------------------------------------- whole FP32 layer
@pytest.mark.parametrize("spec_idx", range(len(wl.LAYER_LIST)))
def test_layer_list_shapes_vs_torch(spec_idx):
    """Every list layer's shape (spatial size cut to at most 24 so the check is
    quick) against torch float64; the result is the float32 rounding of it."""
    spec = wl.LAYER_LIST[spec_idx]
    small = wl.LayerSpec(spec.c_in, spec.c_out, spec.k, spec.stride, min(spec.h, 24))
    x, p = wl.layer_inputs(small, 2, seed=0, layer_index=spec_idx)
    y = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, small.stride, small.pad)
    ref, _ = torch_layer(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, small.stride, small.pad)
    assert y.shape == ref.shape == (2, small.c_out, small.oh, small.ow)
    np.testing.assert_allclose(y, ref.astype(np.float32), rtol=2e-7, atol=1e-7)


def test_single_layer_full_size_vs_torch():
    spec = wl.SINGLE_LAYER
    x, p = wl.layer_inputs(spec, 1)
    y, work = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad,
                                      return_f64=True)
    ref, _ = torch_layer(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad)
    np.testing.assert_allclose(work, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(y, work.astype(np.float32))


def test_conv_bias_path_vs_torch():
    r = rng(7)
    x = f32(r.standard_normal((1, 3, 9, 9)))
    w = f32(r.standard_normal((4, 3, 3, 3)))
    cb = f32(r.standard_normal(4))
    z = oracle.conv2d(x, w, 2, 1, conv_bias=cb)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x.astype(np.float64)), torch.from_numpy(w.astype(np.float64)),
                                     torch.from_numpy(cb.astype(np.float64)), stride=2, padding=1).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-13)



# ------------------------------------------ activation and residual (plain conv + bias, residual add)
def _identity_bn(c):
    """BN that is exactly the identity: var + eps == 1 in float32 (eps = 2^-10)."""
    eps = 2.0 ** -10
    return (np.ones(c, np.float32), np.zeros(c, np.float32), np.zeros(c, np.float32),
            np.full(c, 1.0 - eps, np.float32), eps)


def _delta_kernel(c, k):
    w = np.zeros((c, c, k, k), np.float32)
    for i in range(c):
        w[i, i, k // 2, k // 2] = 1.0
    return w


def test_act_silu_without_residual_is_the_fused_layer():
    spec = wl.LayerSpec(8, 12, 3, 2, 11)
    x, p = wl.layer_inputs(spec, 2, layer_index=3)
    a = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 2, 1)
    b = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 2, 1, act=0)
    assert np.array_equal(a.view(np.int32), b.view(np.int32))


@pytest.mark.parametrize("k", [1, 3, 5])
def test_identity_act_delta_kernel_identity_bn_returns_input(k):
    r = rng(11)
    x = f32(r.standard_normal((2, 5, 7, 9)))
    g, b, m, v, eps = _identity_bn(5)
    y = oracle.conv_bn_act_f32(x, _delta_kernel(5, k), g, b, m, v, eps, 1, k // 2, act=1)
    assert np.array_equal(y, x)
    # the same with SiLU is SiLU of the input (closed form, double)
    ys = oracle.conv_bn_act_f32(x, _delta_kernel(5, k), g, b, m, v, eps, 1, k // 2, act=0)
    xd = x.astype(np.float64)
    np.testing.assert_array_equal(ys, (xd / (1.0 + np.exp(-xd))).astype(np.float32))


def test_residual_is_added_after_the_activation():
    r = rng(12)
    x = f32(r.standard_normal((1, 4, 6, 6)))
    res = f32(r.standard_normal((1, 4, 6, 6)))
    g, b, m, v, eps = _identity_bn(4)
    # identity everything: y = x + r, rounded once (exactly numpy's float32 add)
    y = oracle.conv_bn_act_f32(x, _delta_kernel(4, 3), g, b, m, v, eps, 1, 1, act=1, residual=res)
    assert np.array_equal(y, x + res)
    # a real layer: y = float(SiLU(BN(conv)) in double + r)
    spec = wl.LayerSpec(6, 10, 3, 1, 8)
    x2, p = wl.layer_inputs(spec, 2, layer_index=5)
    r2 = f32(r.standard_normal((2, 10, 8, 8)))
    _, work = oracle.conv_bn_silu_f32(x2, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1, return_f64=True)
    y2 = oracle.conv_bn_act_f32(x2, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1, act=0, residual=r2)
    assert np.array_equal(y2, (work + r2.astype(np.float64)).astype(np.float32))


def test_identity_act_vs_torch():
    """Plain conv + BN (no SiLU) against torch float64 conv2d + batch_norm."""
    spec = wl.LayerSpec(16, 24, 3, 2, 13)
    x, p = wl.layer_inputs(spec, 2, layer_index=6)
    y, work = oracle.conv_bn_act_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 2, 1, act=1, return_f64=True)
    t = torch.nn.functional.conv2d(torch.from_numpy(x.astype(np.float64)), torch.from_numpy(p.w.astype(np.float64)),
                                   stride=2, padding=1)
    ref = torch.nn.functional.batch_norm(t, torch.from_numpy(p.mean.astype(np.float64)),
                                         torch.from_numpy(p.var.astype(np.float64)),
                                         torch.from_numpy(p.gamma.astype(np.float64)),
                                         torch.from_numpy(p.beta.astype(np.float64)), False, 0.0,
                                         float(np.float32(p.eps))).numpy()
    np.testing.assert_allclose(work, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------ INT8
def _ulp_distance(a, b):
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, np.int64(-2**31) - ia, ia)
    ib = np.where(ib < 0, np.int64(-2**31) - ib, ib)
    return np.abs(ia - ib)


def test_spec_exp_within_2ulp():
    r = rng(8)
    xs = np.concatenate([
        f32(r.uniform(-87.0, 88.0, 3_000_000)),
        f32(r.uniform(-1.0, 1.0, 1_000_000)),
        f32(np.linspace(-87.0, 88.0, 1_000_001)),
        f32(r.uniform(-1e-3, 1e-3, 100_000)),
    ])
    y = oracle.spec_exp(xs)
    ref = np.exp(xs.astype(np.float64)).astype(np.float32)
    d = _ulp_distance(y, ref)
    assert d.max() <= 2, (d.max(), xs[np.argmax(d)])


def test_spec_exp_special_points():
    y = oracle.spec_exp(f32([0.0, 88.5, 100.0, -87.5, -200.0, 1.0, -1.0]))
    assert y[0] == 1.0
    assert np.isinf(y[1]) and np.isinf(y[2]) and y[1] > 0
    assert y[3] == 0.0 and y[4] == 0.0
    assert _ulp_distance(y[5:6], f32([math.e]))[0] <= 1
    assert _ulp_distance(y[6:7], f32([1 / math.e]))[0] <= 1


def test_round_half_even_ties():
    x = f32([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.5, 200.0, -128.5, -300.0, 3.49, -3.51])
    q = oracle.quantize_act(x, 1.0)
    assert q.tolist() == [0, 2, 2, 0, -2, -2, 126, 127, 127, -128, -128, 3, -4]


def test_s_x_is_the_normal_percentile():
    from scipy.special import erfc, erfcinv
    t = math.sqrt(2.0) * erfcinv(1e-5)
    assert abs(t - wl.ABS_NORMAL_P99999) < 1e-9
    assert abs(erfc(wl.ABS_NORMAL_P99999 / math.sqrt(2)) - 1e-5) < 1e-12


def test_fold_quant_invariants():
    spec = wl.LayerSpec(8, 6, 3, 1, 5)
    _, p = wl.layer_inputs(spec, 1, layer_index=3)
    w = p.w.copy()
    w[4] = 0.0                                      # an all-zero channel
    s_x = float(wl.S_X_INT8)
    q_w, bias, m_c = oracle.fold_quant_i8(w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x)
    s = p.gamma.astype(np.float64) / np.sqrt(p.var.astype(np.float64) + np.float64(np.float32(p.eps)))
    wf = w.reshape(6, -1).astype(np.float64) * s[:, None]
    bf = p.beta.astype(np.float64) - p.mean.astype(np.float64) * s
    s_w = m_c.astype(np.float64) / np.float64(np.float32(s_x))
    for c in range(6):
        q = q_w[c].reshape(-1).astype(np.float64)
        if c == 4:
            assert np.all(q == 0) and abs(s_w[c] - 1.0) < 1e-6
            continue
        assert np.abs(q).max() == 127
        assert np.all(np.abs(q * s_w[c] - wf[c]) <= 0.5 * s_w[c] * (1 + 1e-5))
    assert np.all(np.abs(bias * m_c.astype(np.float64) - bf) <= 0.5 * m_c * (1 + 1e-5))


@pytest.mark.parametrize("k,stride", [(1, 1), (3, 1), (3, 2)])
def test_int8_accumulation_exact(k, stride):
    r = rng(20 + k + stride)
    q_x = r.integers(-128, 128, size=(2, 7, 9, 9)).astype(np.int8)
    q_w = r.integers(-127, 128, size=(5, 7, k, k)).astype(np.int8)
    bias = r.integers(-10**6, 10**6, size=5).astype(np.int32)
    m_c = np.full(5, 1e-3, np.float32)
    q_y, acc = oracle.conv_i8(q_x, q_w, bias, m_c, 0.05, stride, k // 2, return_acc=True)
    ref = torch.nn.functional.conv2d(torch.from_numpy(q_x.astype(np.float64)),
                                     torch.from_numpy(q_w.astype(np.float64)), stride=stride, padding=k // 2).numpy()
    assert np.array_equal(acc.astype(np.int64), ref.astype(np.int64) + bias[None, :, None, None])


def test_int8_worst_case_accumulator_fits():
    """|acc| <= 2304*128*127 for the widest layer (256 channels, 3x3)."""
    q_x = np.full((1, 256, 3, 3), -128, np.int8)
    q_w = np.full((1, 256, 3, 3), 127, np.int8)
    _, acc = oracle.conv_i8(q_x, q_w, np.zeros(1, np.int32), np.ones(1, np.float32), 1.0, 1, 1, return_acc=True)
    assert acc[0, 0, 1, 1] == -2304 * 128 * 127


def test_requant_against_float64():
    r = rng(9)
    accs = r.integers(-200000, 200000, size=20000)
    m_c, s_y = 1.7e-4, 0.031
    inv = float(np.float32(1.0) / np.float32(s_y))
    got = np.array([oracle.requant(int(a), m_c, inv) for a in accs])
    t = accs.astype(np.float64) * np.float64(np.float32(m_c))
    v = np.clip(t / (1 + np.exp(-t)) * inv, -128, 127)
    want = np.round(v)   # numpy rounds half to even
    near_tie = np.abs(v - np.floor(v) - 0.5) < 1e-4
    assert np.all(np.abs(got - want) <= 1)
    assert np.all(got[~near_tie] == want[~near_tie])


def test_requant_edges():
    inv = 1.0 / 0.05
    assert oracle.requant(0, 0.01, inv) == 0
    assert oracle.requant(-10**7, 0.01, inv) == 0        # t <= -88: SiLU underflows to -0
    assert oracle.requant(10**7, 0.01, inv) == 127       # saturates
    assert oracle.requant(-128, 0.01, inv) == -6          # SiLU(-1.28) = -0.27846; x20 = -5.57


def test_int8_layer_tracks_fp32_layer():
    spec = wl.LayerSpec(16, 8, 3, 1, 12)
    x, p = wl.layer_inputs(spec, 2, layer_index=5)
    s_x = float(wl.S_X_INT8)
    y32 = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1)
    s_y = float(np.float32(np.abs(y32).max() / 127))
    q_x = oracle.quantize_act(x, s_x)
    q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x)
    q_y = oracle.conv_i8(q_x, q_w, bias, m_c, s_y, 1, 1)
    err = np.abs(q_y.astype(np.float64) * s_y - y32)
    assert err.mean() < 1.0 * s_y and err.max() < 6 * s_y


# ------------------------------------------------- asymmetric INT8 activations
# ("Edge optimisation of YOLO26", Design notes: asymmetric activations,
# symmetric per-channel weights; the affine scheme r = s (q - z).)

@pytest.mark.parametrize("k,stride,z_x", [(3, 1, -37), (3, 2, 90), (1, 1, -128), (5, 2, 127)])
def test_int8_zero_point_accumulation_exact(k, stride, z_x):
    """acc = bias + conv(q_x - z_x, q_w) with zero padding in the (q - z)
    domain: a padded tap is a real zero and adds nothing.  PyTorch float64
    conv2d (exact on these integers) is the independent sum."""
    r = rng(40 + k + stride)
    q_x = r.integers(-128, 128, size=(2, 6, 9, 11)).astype(np.int8)
    q_w = r.integers(-127, 128, size=(4, 6, k, k)).astype(np.int8)
    bias = r.integers(-10**5, 10**5, size=4).astype(np.int32)
    m_c = np.full(4, 1e-4, np.float32)
    _, acc = oracle.conv_i8(q_x, q_w, bias, m_c, 0.05, stride, k // 2, return_acc=True, z_x=z_x, z_y=3)
    xs = torch.from_numpy(q_x.astype(np.float64) - z_x)
    ref = torch.nn.functional.conv2d(xs, torch.from_numpy(q_w.astype(np.float64)), stride=stride,
                                     padding=k // 2).numpy()
    assert np.array_equal(acc.astype(np.int64), ref.astype(np.int64) + bias[None, :, None, None])


def test_quantize_zero_point():
    """q = clamp(rne(x / s) + z): x = 0 maps to z, the dequantised value
    s (q - z) is within s/2 of x inside the range, and the ends saturate."""
    s = 0.02
    for z in (-128, -61, 0, 44, 127):
        lo, hi = (-128 - z) * s, (127 - z) * s
        x = np.linspace(lo + s, hi - s, 4001, dtype=np.float32)
        q = oracle.quantize_act(np.concatenate([x, [0.0, lo - 1, hi + 1]]).astype(np.float32), s, z)
        assert q[-3] == z and q[-2] == -128 and q[-1] == 127
        err = np.abs(s * (q[:-3].astype(np.float64) - z) - x)
        assert err.max() <= 0.5 * s * (1 + 1e-4)


def test_requant_zero_point_against_float64():
    r = rng(11)
    accs = r.integers(-200000, 200000, size=20000)
    m_c, s_y = 1.7e-4, 0.031
    inv = float(np.float32(1.0) / np.float32(s_y))
    for z_y in (-100, 57):
        got = np.array([oracle.requant(int(a), m_c, inv, z_y) for a in accs])
        t = accs.astype(np.float64) * np.float64(np.float32(m_c))
        v = t / (1 + np.exp(-t)) * inv
        want = np.clip(np.round(v) + z_y, -128, 127)   # numpy rounds half to even
        near_tie = np.abs(v - np.floor(v) - 0.5) < 1e-4
        assert np.all(np.abs(got - want) <= 1)
        assert np.all(got[~near_tie] == want[~near_tie])
        assert oracle.requant(0, m_c, inv, z_y) == z_y


def test_asymmetric_int8_layer_tracks_fp32_layer():
    """Post-SiLU-like activations (mostly positive) quantised with a zero
    point near the bottom of the code range: the dequantised output of the
    asymmetric layer follows the FP32 layer within a few output steps."""
    spec = wl.LayerSpec(16, 8, 3, 1, 12)
    x, p = wl.layer_inputs(spec, 2, layer_index=6)
    x = (x / (1 + np.exp(-x))).astype(np.float32)          # SiLU(x): in [-0.28, ...)
    s_x = float(np.float32((x.max() - x.min()) / 255))
    z_x = int(-128 - round(float(x.min()) / s_x))
    y32 = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, 1, 1)
    s_y = float(np.float32((y32.max() - y32.min()) / 255))
    z_y = int(-128 - round(float(y32.min()) / s_y))
    q_x = oracle.quantize_act(x, s_x, z_x)
    q_w, bias, m_c = oracle.fold_quant_i8(p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x)
    q_y = oracle.conv_i8(q_x, q_w, bias, m_c, s_y, 1, 1, z_x=z_x, z_y=z_y)
    err = np.abs((q_y.astype(np.float64) - z_y) * s_y - y32)
    assert err.mean() < 1.0 * s_y and err.max() < 6 * s_y


# ------------------------------------------------------------ max pooling glue

@pytest.mark.parametrize("k,stride,pad,hw", [(5, 1, 2, (13, 17)), (3, 2, 1, (12, 9)), (2, 2, 0, (8, 10)),
                                             (3, 1, 0, (5, 5)), (5, 1, 2, (1, 1))])
def test_maxpool_vs_torch(k, stride, pad, hw):
    """Against PyTorch's max_pool2d (padding takes no part, floor size)."""
    x = rng(50 + k).standard_normal((2, 5) + hw).astype(np.float32)
    got = oracle.maxpool2d_f32(x, k, stride, pad)
    want = torch.nn.functional.max_pool2d(torch.from_numpy(x), k, stride, pad).numpy()
    assert got.shape == want.shape and np.array_equal(got, want)


def test_maxpool_padding_takes_no_part_and_nan_propagates():
    x = -np.ones((1, 1, 3, 3), np.float32) * 5      # all negative: a zero-padded window would give 0
    assert np.all(oracle.maxpool2d_f32(x, 3, 1, 1) == -5)
    x[0, 0, 1, 1] = np.nan
    assert np.isnan(oracle.maxpool2d_f32(x, 3, 1, 1)).all()


# ------------------------------------------------------------ INT8 seams
def test_round_bf16_matches_torch_conversion():
    """oracle.round_bf16 against torch's float32 -> bfloat16 conversion (a
    library routine, round to nearest even), on random magnitudes, on exact
    ties with even and odd kept parts, subnormals, infinities and zero."""
    import torch
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 120, 200000))).astype(np.float32)
    ties = np.array([0x3f808000, 0x3f818000, 0xbf808000, 0xbf818000, 0x3f80ffff, 0x3f807fff,
                     0x00008000, 0x00018000, 0x7f7f8000, 0x00000001], dtype=np.uint32).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -3e-39], dtype=np.float32)
    x = np.concatenate([x, ties, special])
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = oracle.round_bf16(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    nan = oracle.round_bf16(np.array([np.nan], np.float32))
    assert np.isnan(nan).all()


def test_dequantize_power_of_two_scale_is_exact():
    """With s = 2^k the product (q - z) * s is exact: the closed form in
    integer arithmetic."""
    q = np.arange(-128, 128, dtype=np.int8)
    for k in (-7, -1, 0, 3):
        for z in (0, -128, 17, 127):
            got = oracle.dequantize_i8(q, float(2.0 ** k), z)
            want = np.array([(int(v) - z) * 2.0 ** k for v in q])
            assert np.array_equal(got.astype(np.float64), want)


def test_dequantize_inverts_the_quantiser():
    """dequantize(quantize(x)) is within half a step of x wherever the
    quantiser does not saturate: scale and zero point mean the same thing
    on both sides of a seam (a sign or offset slip fails this)."""
    rng = np.random.default_rng(5)
    for s, z in ((0.0347809, 0), (0.05, -40), (0.013, 90)):
        lo, hi = (-128 - z + 0.5) * s, (127 - z - 0.5) * s
        x = rng.uniform(lo, hi, 100000).astype(np.float32)
        r = oracle.dequantize_i8(oracle.quantize_act(x, s, z), s, z)
        assert np.max(np.abs(r.astype(np.float64) - x)) <= s / 2 * (1 + 1e-5)
