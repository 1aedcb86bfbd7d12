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


def max_scaled_err(got, ref) -> float:
    """Max abs error at unit output scale, for NCHW tensors:
    max |got - ref| / max(1, |ref|, rms_c(ref)), rms_c = the RMS of the
    element's output channel.  The layer's BatchNorm gives each channel its
    own scale (gamma / sqrt(var) up to ~2), and a bfloat16 output alone
    carries a relative rounding of up to 2^-9; dividing by the channel scale
    brings every channel to unit scale before the absolute bound applies."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if not np.size(ref):
        return 0.0
    axes = tuple(i for i in range(ref.ndim) if i != 1)
    rms_c = np.sqrt(np.mean(ref * ref, axis=axes, keepdims=True))
    den = np.maximum(np.maximum(1.0, np.abs(ref)), rms_c)
    return float(np.max(np.abs(got - ref) / den))


# FP32 CUDA-core path: relative L2 <= 1e-5.  TF32/BF16 tensor-core paths:
# relative L2 <= 5e-3 and max abs <= 2e-2 on unit-scale outputs (checked as
# max |err| / max(1, |ref|, channel RMS) <= 2e-2).  INT8: exact.
TOL_FP32_REL_L2 = 1e-5
TOL_TC_REL_L2 = 5e-3
TOL_TC_MAX_ABS = 2e-2
