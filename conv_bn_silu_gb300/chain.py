"""The 40-layer whole-frame chain of fused layers (YOLO26n-scale shapes).

Layers and their sources are those of `workloads.chain_layers()`: the list's
first eleven layers from the frame, the 384->128 1x1 layer on
concat(upsample2x(layer 10), layer 7), and 28 stride-1 repeats at 80/40/20.
Every computation runs in libcbs.so: the chain-entry layout step
(cbs_pack_input), the fused layers and the neck glue.  Layer 11 is a
two-input layer: it reads the upsampled layer 10 and layer 7 straight from
their buffers (the channel concatenation happens in its input loads), so the
only glue kernel is the 2x upsample.

FP32 runs in NCHW by default, on the CUDA cores; with layout=NHWC its layers
take the 3xTF32 tensor-core variant (the FP32 bar).  TF32, BF16 and INT8 run
the tensor-core variants in NHWC.  In NHWC only the frame needs packing.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _binding as B
from . import workloads as wl
from .layer import FusedConvBnSilu, current_stream, make_desc

PRECS = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16}


class Chain:
    def __init__(self, prec: str, n: int, seed: int = 0, device="cuda", layout: int | None = None):
        self.prec = prec
        self.n = n
        self.device = torch.device(device)
        self.specs = wl.chain_layers()
        cp = PRECS[prec]
        if layout is None:
            layout = B.CBS_NCHW if prec == "fp32" else B.CBS_NHWC
        if prec != "fp32" and layout != B.CBS_NHWC:
            raise ValueError("the tensor-core precisions run the chain in NHWC")
        self.layout = layout
        self.layers = []
        for i, cl in enumerate(self.specs):
            s = cl.spec
            p = wl.layer_params(s, seed=seed, layer_index=100 + i)
            c_in_b = self.specs[cl.src[2]].spec.c_out if cl.src[0] == "upcat" else 0
            desc = make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad, prec=cp,
                             in_layout=self.layout, out_layout=self.layout, c_in_b=c_in_b)
            self.layers.append(FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps,
                                               device=self.device))
        self.outs = [layer.empty_y() for layer in self.layers]
        self.x0 = self.layers[0].empty_x()
        self.glue = self.layers[11].empty_x()   # upsample2x(layer 10): the first input of layer 11

    def params(self, i: int, seed: int = 0):
        return wl.layer_params(self.specs[i].spec, seed=seed, layer_index=100 + i)

    def input_of(self, i: int):
        """The device tensor layer i reads (its first input; after its source has run)."""
        src = self.specs[i].src
        if src[0] == "frame":
            return self.x0
        if src[0] == "layer":
            return self.outs[src[1]]
        return self.glue

    def second_input_of(self, i: int):
        """The second input of a two-input layer, else None."""
        src = self.specs[i].src
        return self.outs[src[2]] if src[0] == "upcat" else None

    def launches_per_frame(self) -> int:
        return len(self.layers) + 2  # 40 fused layers, frame packing, one upsample kernel

    def run(self, frame_nchw: torch.Tensor, stream: int | None = None):
        """One frame batch: pack the frame, then the 40 layers in order."""
        s = current_stream() if stream is None else stream
        B.cbs_pack_input(self.layers[0].plan, frame_nchw, self.x0, 0.0, s)
        for i, layer in enumerate(self.layers):
            src = self.specs[i].src
            if src[0] == "upcat":
                a = self.outs[src[1]]
                if self.layout == B.CBS_NHWC:
                    n, h, w, ca = a.shape
                else:
                    n, ca, h, w = a.shape
                B.cbs_upsample2x_concat(a, ca, None, 0, self.glue, n, 2 * h, 2 * w, self.layout, a.element_size(), s)
            layer(self.input_of(i), self.outs[i], stream=s, x_b=self.second_input_of(i))
        return self.outs

    def flops(self) -> int:
        return sum(cl.spec.flops(self.n) for cl in self.specs)

    def alg_bytes(self, act_bytes: int) -> int:
        return sum(cl.spec.alg_bytes(self.n, act_bytes) for cl in self.specs)


def to_nchw_numpy(t: torch.Tensor, layout: int) -> np.ndarray:
    a = t.float().cpu().numpy()
    return np.ascontiguousarray(a.transpose(0, 3, 1, 2)) if layout == B.CBS_NHWC else a
