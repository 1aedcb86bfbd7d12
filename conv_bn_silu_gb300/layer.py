"""Torch-facing helpers over the C ABI: device buffers from PyTorch's caching
allocator, the current CUDA stream, and the calls of include/cbs.h.

Nothing here computes: packing, folding and the fused layer all run in
libcbs.so's kernels.
"""
from __future__ import annotations

import copy
import torch

from . import _binding as B
from . import tuning

_TORCH_DTYPE = {B.CBS_FP32: torch.float32, B.CBS_TF32: torch.float32,
                B.CBS_BF16: torch.bfloat16, B.CBS_INT8: torch.int8}


def current_stream() -> int:
    return torch.cuda.current_stream().cuda_stream


_sms_cache = {}


def device_sms() -> int:
    """SM count of the current CUDA device (0 without one: the plan then
    assumes the GB300's 152)."""
    if not torch.cuda.is_available():
        return 0
    dev = torch.cuda.current_device()
    if dev not in _sms_cache:
        _sms_cache[dev] = int(torch.cuda.get_device_properties(dev).multi_processor_count)
    return _sms_cache[dev]


def make_desc(n, c_in, h, w, c_out, k, stride, pad=None, prec=B.CBS_FP32, in_layout=None,
              out_layout=None, force_variant=-1, force_split_k=0, force_block_n=0,
              force_block_m=0, out_row_stride=0, force_k_group=0, force_b_resident=0,
              force_window=0, activation=B.CBS_ACT_SILU, residual=0, c_in_b=0, zero_point_x=0,
              zero_point_y=0, num_sms=None, force_issuer_split=0) -> B.cbs_layer_desc:
    """A layer descriptor; num_sms defaults to the current device's SM count."""
    if num_sms is None:
        num_sms = device_sms()
    if pad is None:
        pad = k // 2
    if in_layout is None:
        in_layout = B.CBS_NCHW if prec == B.CBS_FP32 else B.CBS_NHWC
    if out_layout is None:
        out_layout = in_layout
    d = B.cbs_layer_desc()
    for name, v in dict(n=n, c_in=c_in, h=h, w=w, c_out=c_out, k=k, stride=stride, pad=pad,
                        in_layout=in_layout, out_layout=out_layout, prec=prec,
                        force_variant=force_variant, force_split_k=force_split_k,
                        force_block_n=force_block_n, force_block_m=force_block_m,
                        out_row_stride=out_row_stride, force_k_group=force_k_group,
                        force_b_resident=force_b_resident, force_window=force_window,
                        activation=activation, residual=residual, c_in_b=c_in_b, zero_point_x=zero_point_x,
                        zero_point_y=zero_point_y, num_sms=num_sms,
                        force_issuer_split=force_issuer_split).items():
        setattr(d, name, int(v))
    return d


def _dev_f32(a, device):
    t = torch.as_tensor(a, dtype=torch.float32)
    return t.to(device).contiguous()


class FusedConvBnSilu:
    """One planned layer with its folded weights resident on the device."""

    def __init__(self, desc: B.cbs_layer_desc, w, gamma, beta, mean, var, eps: float,
                 conv_bias=None, s_x: float = 0.0, device="cuda", tuned: bool = True):
        """tuned: take the measured configuration of tuning.py's table when
        the shape is in it and `desc` forces nothing."""
        self.device = torch.device(device)
        self.desc = tuning.tuned_desc(desc) if tuned else desc
        desc = self.desc
        self.plan = B.cbs_plan(desc)
        self.prec = desc.prec
        self.s_x = float(s_x)
        p = self.plan
        self.w_packed = torch.empty(p.w_packed_bytes, dtype=torch.uint8, device=self.device)
        self.bias = torch.empty(p.bias_bytes, dtype=torch.uint8, device=self.device)
        self.m_c = (torch.empty(desc.c_out, dtype=torch.float32, device=self.device)
                    if self.prec == B.CBS_INT8 else None)
        ws = max(int(p.workspace_bytes), 0)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device) if ws else None
        s = current_stream()
        raw = [_dev_f32(a, self.device) for a in (w, gamma, beta, mean, var)]
        cb = None if conv_bias is None else _dev_f32(conv_bias, self.device)
        B.cbs_fold_bn(p, raw[0], cb, raw[1], raw[2], raw[3], raw[4], float(eps), self.s_x,
                      self.w_packed, self.bias, self.m_c, s)
        if self.workspace is not None:
            B.cbs_workspace_init(self.workspace, int(p.workspace_bytes), s)
        self._keep = (raw, cb)  # inputs of the asynchronous fold stay alive

    def fork(self) -> "FusedConvBnSilu":
        """The same layer (plan, folded weights and bias shared) with a
        split-K workspace of its own, for calls that may run at the same time
        as this layer's on another stream: two launches sharing one workspace
        would mix their partial tiles and arrival counters."""
        twin = copy.copy(self)
        if self.workspace is not None:
            twin.workspace = torch.empty_like(self.workspace)
            B.cbs_workspace_init(twin.workspace, int(self.plan.workspace_bytes), current_stream())
        return twin

    # ---------------------------------------------------------------- shapes
    @property
    def x_dtype(self):
        return _TORCH_DTYPE[self.prec]

    def x_shape(self):
        """Shape of x (of the first input, for a two-input layer)."""
        d, p = self.desc, self.plan
        c_a = d.c_in - d.c_in_b
        if d.in_layout == B.CBS_NCHW:
            return (d.n, c_a, d.h, d.w)
        return (d.n, d.h, d.w, c_a if d.c_in_b else p.c_in_pad)

    def x_b_shape(self):
        """Shape of x_b, the second input of a two-input layer."""
        d, p = self.desc, self.plan
        assert d.c_in_b > 0
        if d.in_layout == B.CBS_NCHW:
            return (d.n, d.c_in_b, d.h, d.w)
        return (d.n, d.h, d.w, p.c_in_pad - (d.c_in - d.c_in_b))

    def y_shape(self):
        d, p = self.desc, self.plan
        if d.out_layout == B.CBS_NCHW:
            return (d.n, d.c_out, p.oh, p.out_row_stride)
        return (d.n, p.oh, p.ow, d.c_out)

    def empty_x(self):
        return torch.empty(self.x_shape(), dtype=self.x_dtype, device=self.device)

    def empty_y(self):
        return torch.empty(self.y_shape(), dtype=self.x_dtype, device=self.device)

    def empty_x_b(self):
        return torch.empty(self.x_b_shape(), dtype=self.x_dtype, device=self.device)

    # ----------------------------------------------------------------- calls
    def pack_input(self, x_nchw: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        """NCHW float32 device tensor -> the plan's input format (kernel)."""
        assert x_nchw.is_cuda and x_nchw.dtype == torch.float32 and x_nchw.is_contiguous()
        out = self.empty_x() if out is None else out
        B.cbs_pack_input(self.plan, x_nchw, out, self.s_x, current_stream())
        return out

    def pack_inputs(self, x_nchw: torch.Tensor, x_b_nchw: torch.Tensor):
        """Two-input layer: each NCHW float32 input -> its input format, each
        through a one-input plan of its own channel count (kernel)."""
        d = self.desc
        out = []
        for t, shape in ((x_nchw, self.x_shape()), (x_b_nchw, self.x_b_shape())):
            assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
            one = make_desc(d.n, t.shape[1], d.h, d.w, 16, 1, 1, 0, prec=d.prec, in_layout=d.in_layout,
                            force_variant=self.plan.variant, zero_point_x=d.zero_point_x)
            o = torch.empty(shape, dtype=self.x_dtype, device=self.device)
            B.cbs_pack_input(B.cbs_plan(one), t, o, self.s_x, current_stream())
            out.append(o)
        return tuple(out)

    def __call__(self, x: torch.Tensor, y: torch.Tensor | None = None, s_y: float | None = None,
                 stream: int | None = None, residual: torch.Tensor | None = None,
                 x_b: torch.Tensor | None = None) -> torch.Tensor:
        """residual: for descriptors with residual=1, a tensor shaped and typed
        like y, added after the activation (may be y itself).  x_b: the second
        input of a two-input (channel concatenation) layer."""
        y = self.empty_y() if y is None else y
        s = current_stream() if stream is None else stream
        ws_bytes = int(self.plan.workspace_bytes)
        if self.desc.c_in_b and self.prec == B.CBS_INT8:
            assert s_y is not None
            B.cbs_conv_bn_silu_i8_cat(self.plan, x, x_b, self.w_packed, self.bias, self.m_c, float(s_y), y,
                                      self.workspace, ws_bytes, s)
            return y
        if self.desc.c_in_b:
            B.cbs_conv_bn_act_cat(self.plan, x, x_b, self.w_packed, self.bias, residual, y, self.workspace,
                                  ws_bytes, s)
            return y
        if self.desc.residual or self.desc.activation != B.CBS_ACT_SILU:
            B.cbs_conv_bn_act(self.plan, x, self.w_packed, self.bias, residual, y, self.workspace, ws_bytes, s)
            return y
        if self.prec == B.CBS_INT8:
            assert s_y is not None
            B.cbs_conv_bn_silu_i8(self.plan, x, self.w_packed, self.bias, self.m_c, float(s_y), y,
                                  self.workspace, ws_bytes, s)
        else:
            B.cbs_conv_bn_silu_f32(self.plan, x, self.w_packed, self.bias, y, self.workspace,
                                   ws_bytes, s)
        return y


_PREC_OF_DTYPE = {torch.float32: B.CBS_FP32, torch.bfloat16: B.CBS_BF16, torch.int8: B.CBS_INT8}


def maxpool2d(x: torch.Tensor, k: int, stride: int, pad: int, layout: int, out: torch.Tensor | None = None):
    """Max pooling (the SPPF glue), in the given layout (kernel)."""
    if layout == B.CBS_NHWC:
        n, h, w, c = x.shape
    else:
        n, c, h, w = x.shape
    oh, ow = (h + 2 * pad - k) // stride + 1, (w + 2 * pad - k) // stride + 1
    shape = (n, oh, ow, c) if layout == B.CBS_NHWC else (n, c, oh, ow)
    out = torch.empty(shape, dtype=x.dtype, device=x.device) if out is None else out
    B.cbs_maxpool2d(x, out, n, c, h, w, k, stride, pad, layout, _PREC_OF_DTYPE[x.dtype], current_stream())
    return out


def sppf_pool(x: torch.Tensor, k: int, layout: int, out: torch.Tensor | None = None):
    """The SPPF block's three chained k x k stride-1 max pools of x, side by
    side along channels (kernel)."""
    if layout == B.CBS_NHWC:
        n, h, w, c = x.shape
        shape = (n, h, w, 3 * c)
    else:
        n, c, h, w = x.shape
        shape = (n, 3 * c, h, w)
    out = torch.empty(shape, dtype=x.dtype, device=x.device) if out is None else out
    B.cbs_sppf_pool(x, out, n, c, h, w, k, layout, _PREC_OF_DTYPE[x.dtype], current_stream())
    return out


def upsample2x(a: torch.Tensor, layout: int, out: torch.Tensor | None = None):
    """Nearest 2x upsample (the glue in front of a two-input layer)."""
    if layout == B.CBS_NHWC:
        n, h, w, ca = a.shape
        shape = (n, 2 * h, 2 * w, ca)
    else:
        n, ca, h, w = a.shape
        shape = (n, ca, 2 * h, 2 * w)
    out = torch.empty(shape, dtype=a.dtype, device=a.device) if out is None else out
    B.cbs_upsample2x_concat(a, ca, None, 0, out, n, 2 * h, 2 * w, layout, a.element_size(), current_stream())
    return out


def upsample2x_concat(a: torch.Tensor, b: torch.Tensor, layout: int, out: torch.Tensor | None = None):
    """Neck glue: concat(upsample2x(a), b) along channels, in the given layout."""
    if layout == B.CBS_NHWC:
        n, h, w, cb = b.shape
        ca = a.shape[3]
        shape = (n, h, w, ca + cb)
    else:
        n, cb, h, w = b.shape
        ca = a.shape[1]
        shape = (n, ca + cb, h, w)
    out = torch.empty(shape, dtype=b.dtype, device=b.device) if out is None else out
    B.cbs_upsample2x_concat(a, ca, b, cb, out, n, h, w, layout, b.element_size(), current_stream())
    return out
