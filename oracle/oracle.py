"""ctypes front end of the C oracle (oracle/cbs_oracle.c).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function takes
and returns numpy arrays in the pages' plain layouts: activations NCHW,
weights OIHW ([C_out, C_in, kH, kW]), as on page 1 of "YOLO26N Inference
Optimisation", section "Weight layout".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        F = ctypes.c_float
        Z = ctypes.c_size_t
        lib.oracle_out_dim.argtypes = [I, I, I, I]
        lib.oracle_out_dim.restype = I
        lib.oracle_conv2d.argtypes = [P, P, P, I, I, I, I, I, I, I, I, P]
        lib.oracle_batchnorm.argtypes = [P, P, P, P, P, F, I, I, Z]
        lib.oracle_silu.argtypes = [P, Z]
        lib.oracle_conv_bn_silu_f32.argtypes = [P, P, P, P, P, P, P, F, I, I, I, I, I, I, I, I, P, P]
        lib.oracle_conv_bn_act_f32.argtypes = [P, P, P, P, P, P, P, F, I, I, I, I, I, I, I, I, I, P, P, P]
        lib.oracle_spec_exp.argtypes = [F]
        lib.oracle_spec_exp.restype = F
        lib.oracle_spec_exp_array.argtypes = [P, P, Z]
        lib.oracle_quantize_act.argtypes = [P, Z, F, P]
        lib.oracle_fold_quant_i8.argtypes = [P, P, P, P, P, F, F, I, I, P, P, P]
        lib.oracle_requant.argtypes = [ctypes.c_int32, F, F]
        lib.oracle_requant.restype = ctypes.c_int8
        lib.oracle_conv_i8.argtypes = [P, P, P, P, F, I, I, I, I, I, I, I, I, P, P]
        lib.oracle_conv_i8.restype = I
        lib.oracle_maxpool2d_f32.argtypes = [P, I, I, I, I, I, I, I, P]
        lib.oracle_set_threads.argtypes = [I]
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = I
        lib.oracle_quantize_act_zp.argtypes = [P, Z, F, I, P]
        lib.oracle_requant_zp.argtypes = [ctypes.c_int32, F, F, I]
        lib.oracle_requant_zp.restype = ctypes.c_int8
        lib.oracle_conv_i8_zp.argtypes = [P, P, P, P, F, I, I, I, I, I, I, I, I, I, I, P, P]
        lib.oracle_conv_i8_zp.restype = I
        lib.oracle_dequantize_i8.argtypes = [P, Z, F, I, P]
        lib.oracle_round_bf16.argtypes = [P, Z, P]
        lib.oracle_requant_zp_array.argtypes = [P, P, Z, F, I, P]
        lib.oracle_spec_exp_max_rel_err.argtypes = [F, F]
        lib.oracle_spec_exp_max_rel_err.restype = ctypes.c_double
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    """Run the oracle's OpenMP loops on n threads (1: single core)."""
    _load().oracle_set_threads(int(n))


def out_dim(size: int, k: int, stride: int, pad: int) -> int:
    return _load().oracle_out_dim(size, k, stride, pad)


def conv2d(x, w, stride: int, pad: int, conv_bias=None) -> np.ndarray:
    """Plain convolution, float inputs, float64 result [N, C_out, OH, OW]."""
    x, w = _f32(x), _f32(w)
    N, C_in, H, W = x.shape
    C_out, C_in2, k, k2 = w.shape
    assert C_in2 == C_in and k2 == k
    OH, OW = out_dim(H, k, stride, pad), out_dim(W, k, stride, pad)
    z = np.empty((N, C_out, OH, OW), np.float64)
    cb = None if conv_bias is None else _f32(conv_bias)
    _load().oracle_conv2d(_ptr(x), _ptr(w), _ptr(cb), N, C_in, H, W, C_out, k, stride, pad, _ptr(z))
    return z


def batchnorm(t, gamma, beta, mean, var, eps: float) -> np.ndarray:
    """Inference BatchNorm on a float64 [N, C, H, W] array (returns a copy)."""
    t = np.array(t, dtype=np.float64, order="C", copy=True)
    N, C = t.shape[:2]
    hw = int(np.prod(t.shape[2:]))
    g, b, m, v = (_f32(a) for a in (gamma, beta, mean, var))
    _load().oracle_batchnorm(_ptr(t), _ptr(g), _ptr(b), _ptr(m), _ptr(v), eps, N, C, hw)
    return t


def silu(t) -> np.ndarray:
    t = np.array(t, dtype=np.float64, order="C", copy=True)
    _load().oracle_silu(_ptr(t), t.size)
    return t


def conv_bn_silu_f32(x, w, gamma, beta, mean, var, eps: float, stride: int, pad: int,
                     conv_bias=None, return_f64: bool = False):
    """y = SiLU(BN(conv(x))) with double arithmetic, rounded once to float32."""
    x, w = _f32(x), _f32(w)
    N, C_in, H, W = x.shape
    C_out, _, k, _ = w.shape
    OH, OW = out_dim(H, k, stride, pad), out_dim(W, k, stride, pad)
    work = np.empty((N, C_out, OH, OW), np.float64)
    y = np.empty((N, C_out, OH, OW), np.float32)
    g, b, m, v = (_f32(a) for a in (gamma, beta, mean, var))
    cb = None if conv_bias is None else _f32(conv_bias)
    _load().oracle_conv_bn_silu_f32(_ptr(x), _ptr(w), _ptr(cb), _ptr(g), _ptr(b), _ptr(m), _ptr(v),
                                    eps, N, C_in, H, W, C_out, k, stride, pad, _ptr(work), _ptr(y))
    return (y, work) if return_f64 else y


def conv_bn_act_f32(x, w, gamma, beta, mean, var, eps: float, stride: int, pad: int, act: int = 0,
                    residual=None, conv_bias=None, return_f64: bool = False):
    """y = act(BN(conv(x))) + residual (act 0: SiLU, 1: identity), double
    arithmetic, rounded once to float32; residual: NCHW, y's shape, or None."""
    x, w = _f32(x), _f32(w)
    N, C_in, H, W = x.shape
    C_out, _, k, _ = w.shape
    OH, OW = out_dim(H, k, stride, pad), out_dim(W, k, stride, pad)
    work = np.empty((N, C_out, OH, OW), np.float64)
    y = np.empty((N, C_out, OH, OW), np.float32)
    g, b, m, v = (_f32(a) for a in (gamma, beta, mean, var))
    cb = None if conv_bias is None else _f32(conv_bias)
    r = None
    if residual is not None:
        r = _f32(residual)
        assert r.shape == y.shape
    _load().oracle_conv_bn_act_f32(_ptr(x), _ptr(w), _ptr(cb), _ptr(g), _ptr(b), _ptr(m), _ptr(v), eps, N,
                                   C_in, H, W, C_out, k, stride, pad, int(act), _ptr(r), _ptr(work), _ptr(y))
    return (y, work) if return_f64 else y


def maxpool2d_f32(x, k: int, stride: int, pad: int) -> np.ndarray:
    """Max pooling of an NCHW float32 array; padding takes no part, floor
    output size, NaN propagates."""
    x = _f32(x)
    N, C, H, W = x.shape
    y = np.empty((N, C, out_dim(H, k, stride, pad), out_dim(W, k, stride, pad)), np.float32)
    _load().oracle_maxpool2d_f32(_ptr(x), N, C, H, W, k, stride, pad, _ptr(y))
    return y


def spec_exp(x) -> np.ndarray:
    """The INT8 epilogue's own exp, elementwise over a float32 array."""
    x = _f32(x)
    y = np.empty_like(x)
    _load().oracle_spec_exp_array(_ptr(x), _ptr(y), x.size)
    return y


def spec_exp_max_rel_err(lo: float, hi: float) -> float:
    """Largest relative error of spec_exp against double exp over every float in [lo, hi]."""
    return float(_load().oracle_spec_exp_max_rel_err(float(lo), float(hi)))


def quantize_act(x, s_x: float, z_x: int = 0) -> np.ndarray:
    """q = clamp(rne(x / s_x), -128, 127); with a zero point z_x (asymmetric
    activations), q = clamp(rne(x / s_x) + z_x, -128, 127)."""
    x = _f32(x)
    q = np.empty(x.shape, np.int8)
    if z_x:
        _load().oracle_quantize_act_zp(_ptr(x), x.size, s_x, int(z_x), _ptr(q))
    else:
        _load().oracle_quantize_act(_ptr(x), x.size, s_x, _ptr(q))
    return q


def dequantize_i8(q, s: float, z: int = 0) -> np.ndarray:
    """r = float(q - z) * s (one float multiply), same shape as q."""
    q = np.ascontiguousarray(q, np.int8)
    r = np.empty(q.shape, np.float32)
    _load().oracle_dequantize_i8(_ptr(q), q.size, float(s), int(z), _ptr(r))
    return r


def round_bf16(x) -> np.ndarray:
    """float32 values rounded to bfloat16 (nearest even), as float32."""
    x = _f32(x)
    out = np.empty_like(x)
    _load().oracle_round_bf16(_ptr(x), x.size, _ptr(out))
    return out


def fold_quant_i8(w, gamma, beta, mean, var, eps: float, s_x: float):
    """Returns (q_w int8 [C_out, C_in, k, k], bias_i32 [C_out], m_c float32 [C_out])."""
    w = _f32(w)
    C_out = w.shape[0]
    kk = int(np.prod(w.shape[1:]))
    q_w = np.empty(w.shape, np.int8)
    bias = np.empty(C_out, np.int32)
    m_c = np.empty(C_out, np.float32)
    g, b, m, v = (_f32(a) for a in (gamma, beta, mean, var))
    _load().oracle_fold_quant_i8(_ptr(w), _ptr(g), _ptr(b), _ptr(m), _ptr(v), eps, s_x,
                                 C_out, kk, _ptr(q_w), _ptr(bias), _ptr(m_c))
    return q_w, bias, m_c


def requant(acc: int, m_c: float, inv_s_y: float, z_y: int = 0) -> int:
    if z_y:
        return int(_load().oracle_requant_zp(int(acc), float(m_c), float(inv_s_y), int(z_y)))
    return int(_load().oracle_requant(int(acc), float(m_c), float(inv_s_y)))


def requant_array(acc, m_c, inv_s_y: float, z_y: int = 0) -> np.ndarray:
    """requant of every (acc[i], m_c[i]) with one inv_s_y and output zero point."""
    acc = np.ascontiguousarray(acc, np.int32)
    m_c = _f32(m_c)
    assert acc.shape == m_c.shape
    q = np.empty(acc.shape, np.int8)
    _load().oracle_requant_zp_array(_ptr(acc), _ptr(m_c), acc.size, float(inv_s_y), int(z_y), _ptr(q))
    return q


def conv_i8(q_x, q_w, bias_i32, m_c, s_y: float, stride: int, pad: int, return_acc: bool = False,
            z_x: int = 0, z_y: int = 0):
    """INT8 layer; returns q_y int8 [N, C_out, OH, OW] (and the int32 accumulators).
    z_x, z_y: zero points of asymmetric input and output codes (0: symmetric)."""
    q_x = np.ascontiguousarray(q_x, np.int8)
    q_w = np.ascontiguousarray(q_w, np.int8)
    bias_i32 = np.ascontiguousarray(bias_i32, np.int32)
    m_c = _f32(m_c)
    N, C_in, H, W = q_x.shape
    C_out, _, k, _ = q_w.shape
    OH, OW = out_dim(H, k, stride, pad), out_dim(W, k, stride, pad)
    q_y = np.empty((N, C_out, OH, OW), np.int8)
    acc = np.empty((N, C_out, OH, OW), np.int32) if return_acc else None
    if z_x or z_y:
        rc = _load().oracle_conv_i8_zp(_ptr(q_x), _ptr(q_w), _ptr(bias_i32), _ptr(m_c), s_y, int(z_x), int(z_y),
                                       N, C_in, H, W, C_out, k, stride, pad, _ptr(q_y), _ptr(acc))
    else:
        rc = _load().oracle_conv_i8(_ptr(q_x), _ptr(q_w), _ptr(bias_i32), _ptr(m_c), s_y,
                                    N, C_in, H, W, C_out, k, stride, pad, _ptr(q_y), _ptr(acc))
    if rc != 0:
        raise OverflowError("INT8 accumulator left the int32 range")
    return (q_y, acc) if return_acc else q_y
