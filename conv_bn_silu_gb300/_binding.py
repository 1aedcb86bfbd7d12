"""ctypes binding of libcbs.so: the C ABI of include/cbs.h under the same names.

Argument marshalling only.  Every computing step runs in the library's CUDA
kernels; there is no Python or CPU fallback, and loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libcbs.so")

CBS_OK = 0
CBS_ERR_INVALID_ARG = -1
CBS_ERR_UNSUPPORTED = -2
CBS_ERR_MISALIGNED = -3
CBS_ERR_WORKSPACE = -4
CBS_ERR_CUDA = -5
CBS_ERR_TIMEOUT = -6
CBS_ERR_PLAN_MISMATCH = -7

CBS_NCHW, CBS_NHWC = 0, 1
CBS_FP32, CBS_TF32, CBS_BF16, CBS_INT8 = 0, 1, 2, 3
CBS_VARIANT_SIMT_FP32, CBS_VARIANT_TC_TF32, CBS_VARIANT_TC_BF16, CBS_VARIANT_TC_INT8 = 0, 1, 2, 3
CBS_VARIANT_STEM = 4
CBS_VARIANT_TC_TF32X3 = 5
CBS_ACT_SILU, CBS_ACT_IDENTITY = 0, 1
CBS_LAUNCH_PDL = 1

EXPORTED = (
    "cbs_plan", "cbs_fold_bn", "cbs_pack_input", "cbs_conv_bn_silu_f32", "cbs_conv_bn_silu_i8",
    "cbs_upsample2x_concat", "cbs_workspace_init", "cbs_read_device_status", "cbs_status_string",
    "cbs_last_error", "cbs_abi_version", "cbs_conv_bn_silu_f32_noalloc", "cbs_conv_bn_act",
    "cbs_conv_bn_act_cat", "cbs_set_launch_options", "cbs_launch_options", "cbs_maxpool2d",
    "cbs_conv_bn_silu_i8_cat", "cbs_selftest_wait_timeout", "cbs_sppf_pool", "cbs_dequantize_i8",
    "cbs_quantize_i8",
)


class cbs_layer_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n", "c_in", "h", "w", "c_out", "k", "stride", "pad", "in_layout", "out_layout", "prec",
        "force_variant", "force_split_k", "force_block_n", "force_block_m", "out_row_stride",
        "force_k_group", "force_b_resident", "force_window", "activation", "residual", "c_in_b",
        "zero_point_x", "zero_point_y", "num_sms", "force_issuer_split")]


class cbs_plan_t(ctypes.Structure):
    _fields_ = [("size", ctypes.c_uint32), ("abi_version", ctypes.c_uint32)] + \
        [(n, ctypes.c_int) for n in (
            "variant", "block_m", "block_n", "block_k", "stages", "split_k", "k_group", "b_resident", "window",
            "issuer_split", "c_in_pad", "k_gemm",
            "oh", "ow", "out_row_stride", "m_tiles", "n_tiles", "grid_ctas", "threads",
            "smem_bytes")] + \
        [(n, ctypes.c_size_t) for n in (
            "x_bytes", "y_bytes", "w_packed_bytes", "bias_bytes", "workspace_bytes", "x_b_bytes")] + \
        [("desc", cbs_layer_desc)]


class CbsError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {status_name(status)} ({status}): {message}")
        self.status = status


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libcbs.so is not built ({LIB_PATH}); run conv_bn_silu_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.cbs_plan.argtypes = [ctypes.POINTER(cbs_layer_desc), ctypes.POINTER(cbs_plan_t)]
        L.cbs_fold_bn.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, P, P, F, F, P, P, P, P]
        L.cbs_pack_input.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, F, P]
        L.cbs_conv_bn_silu_f32.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, P, Z, P]
        L.cbs_conv_bn_act.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, P, P, Z, P]
        L.cbs_conv_bn_act_cat.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, P, P, P, Z, P]
        L.cbs_conv_bn_silu_i8.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, F, P, P, Z, P]
        L.cbs_conv_bn_silu_i8_cat.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, P, F, P, P, Z, P]
        L.cbs_upsample2x_concat.argtypes = [P, I, P, I, P, I, I, I, I, I, P]
        L.cbs_maxpool2d.argtypes = [P, P, I, I, I, I, I, I, I, I, I, P]
        L.cbs_sppf_pool.argtypes = [P, P, I, I, I, I, I, I, I, P]
        L.cbs_dequantize_i8.argtypes = [P, P, Z, F, I, I, P]
        L.cbs_quantize_i8.argtypes = [P, I, P, Z, F, I, P]
        L.cbs_conv_bn_silu_f32_noalloc.argtypes = [ctypes.POINTER(cbs_plan_t), P, P, P, P, P]
        L.cbs_workspace_init.argtypes = [P, Z, P]
        L.cbs_read_device_status.argtypes = [ctypes.POINTER(I), I, P]
        L.cbs_selftest_wait_timeout.argtypes = [I, P]
        L.cbs_status_string.argtypes = [I]
        L.cbs_status_string.restype = ctypes.c_char_p
        L.cbs_last_error.argtypes = []
        L.cbs_last_error.restype = ctypes.c_char_p
        L.cbs_abi_version.argtypes = []
        L.cbs_abi_version.restype = I
        L.cbs_set_launch_options.argtypes = [I]
        L.cbs_launch_options.argtypes = []
        L.cbs_launch_options.restype = I
        for name in EXPORTED:
            if name not in ("cbs_status_string", "cbs_last_error", "cbs_abi_version", "cbs_launch_options"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def status_name(s: int) -> str:
    return lib().cbs_status_string(s).decode()


def _check(status: int, where: str):
    if status != CBS_OK:
        raise CbsError(status, where, lib().cbs_last_error().decode())


def _p(v):
    """Pointer argument: None, an int address, or anything with data_ptr()."""
    if v is None:
        return None
    if isinstance(v, int):
        return v
    return v.data_ptr()


def cbs_abi_version() -> int:
    return lib().cbs_abi_version()


def cbs_status_string(s: int) -> str:
    return status_name(s)


def cbs_last_error() -> str:
    return lib().cbs_last_error().decode()


def cbs_plan(desc: cbs_layer_desc) -> cbs_plan_t:
    plan = cbs_plan_t()
    _check(lib().cbs_plan(ctypes.byref(desc), ctypes.byref(plan)), "cbs_plan")
    return plan


def cbs_fold_bn(plan, w_oihw, conv_bias, gamma, beta, mean, var, eps, s_x, w_packed, bias, m_c,
                stream):
    _check(lib().cbs_fold_bn(ctypes.byref(plan), _p(w_oihw), _p(conv_bias), _p(gamma), _p(beta),
                             _p(mean), _p(var), eps, s_x, _p(w_packed), _p(bias), _p(m_c), stream),
           "cbs_fold_bn")


def cbs_pack_input(plan, x_nchw, x_packed, s_x, stream):
    _check(lib().cbs_pack_input(ctypes.byref(plan), _p(x_nchw), _p(x_packed), s_x, stream),
           "cbs_pack_input")


def cbs_conv_bn_silu_f32(plan, x, w_packed, bias, y, workspace, workspace_bytes, stream):
    _check(lib().cbs_conv_bn_silu_f32(ctypes.byref(plan), _p(x), _p(w_packed), _p(bias), _p(y),
                                      _p(workspace), workspace_bytes, stream),
           "cbs_conv_bn_silu_f32")


def cbs_conv_bn_act(plan, x, w_packed, bias, residual, y, workspace, workspace_bytes, stream):
    _check(lib().cbs_conv_bn_act(ctypes.byref(plan), _p(x), _p(w_packed), _p(bias), _p(residual), _p(y),
                                 _p(workspace), workspace_bytes, stream), "cbs_conv_bn_act")


def cbs_conv_bn_silu_i8_cat(plan, x, x_b, w_packed, bias_i32, m_c, s_y, y, workspace, workspace_bytes, stream):
    _check(lib().cbs_conv_bn_silu_i8_cat(ctypes.byref(plan), _p(x), _p(x_b), _p(w_packed), _p(bias_i32), _p(m_c),
                                         s_y, _p(y), _p(workspace), workspace_bytes, stream), "cbs_conv_bn_silu_i8_cat")


def cbs_maxpool2d(x, y, n, c, h, w, k, stride, pad, layout, prec, stream):
    _check(lib().cbs_maxpool2d(_p(x), _p(y), n, c, h, w, k, stride, pad, layout, prec, stream), "cbs_maxpool2d")


def cbs_sppf_pool(x, y, n, c, h, w, k, layout, prec, stream):
    _check(lib().cbs_sppf_pool(_p(x), _p(y), n, c, h, w, k, layout, prec, stream), "cbs_sppf_pool")


def cbs_dequantize_i8(q, out, count, s, z, out_prec, stream):
    _check(lib().cbs_dequantize_i8(_p(q), _p(out), int(count), float(s), int(z), int(out_prec), stream),
           "cbs_dequantize_i8")


def cbs_quantize_i8(x, in_prec, q, count, s, z, stream):
    _check(lib().cbs_quantize_i8(_p(x), int(in_prec), _p(q), int(count), float(s), int(z), stream), "cbs_quantize_i8")


def cbs_set_launch_options(flags: int):
    _check(lib().cbs_set_launch_options(int(flags)), "cbs_set_launch_options")


def cbs_launch_options() -> int:
    return int(lib().cbs_launch_options())


def cbs_conv_bn_act_cat(plan, x, x_b, w_packed, bias, residual, y, workspace, workspace_bytes, stream):
    _check(lib().cbs_conv_bn_act_cat(ctypes.byref(plan), _p(x), _p(x_b), _p(w_packed), _p(bias), _p(residual),
                                     _p(y), _p(workspace), workspace_bytes, stream), "cbs_conv_bn_act_cat")


def cbs_conv_bn_silu_i8(plan, x, w_packed, bias_i32, m_c, s_y, y, workspace, workspace_bytes,
                        stream):
    _check(lib().cbs_conv_bn_silu_i8(ctypes.byref(plan), _p(x), _p(w_packed), _p(bias_i32),
                                     _p(m_c), s_y, _p(y), _p(workspace), workspace_bytes, stream),
           "cbs_conv_bn_silu_i8")


def cbs_conv_bn_silu_f32_noalloc(plan, x, w_packed, bias, y, stream):
    """FP32 CUDA-core layer with the library's built-in split-K scratch (for
    callers that cannot allocate device memory)."""
    _check(lib().cbs_conv_bn_silu_f32_noalloc(ctypes.byref(plan), _p(x), _p(w_packed), _p(bias), _p(y),
                                              stream), "cbs_conv_bn_silu_f32_noalloc")


def cbs_upsample2x_concat(a, ca, b, cb, out, n, h, w, layout, elem_bytes, stream):
    _check(lib().cbs_upsample2x_concat(_p(a), ca, _p(b), cb, _p(out), n, h, w, layout, elem_bytes,
                                       stream), "cbs_upsample2x_concat")


def cbs_workspace_init(workspace, nbytes, stream):
    _check(lib().cbs_workspace_init(_p(workspace), nbytes, stream), "cbs_workspace_init")


def cbs_read_device_status(reset: bool, stream) -> int:
    out = ctypes.c_int(0)
    _check(lib().cbs_read_device_status(ctypes.byref(out), 1 if reset else 0, stream),
           "cbs_read_device_status")
    return out.value


def cbs_selftest_wait_timeout(limit_us: int, stream):
    """Enqueue the diagnostic kernel whose bounded wait runs out after
    limit_us microseconds and records a timeout in the status word."""
    _check(lib().cbs_selftest_wait_timeout(int(limit_us), stream), "cbs_selftest_wait_timeout")
