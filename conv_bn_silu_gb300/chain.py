"""The 40-layer whole-frame chain of fused layers (YOLO26n-scale shapes),
and the whole synthetic frame (the chain with the SPPF block).

Layers and their sources are those of `workloads.chain_layers()`: the list's
first eleven layers from the frame, the 384->128 1x1 layer on
concat(upsample2x(layer 10), layer 7), and 28 stride-1 repeats at 80/40/20.
Every computation runs in libcbs.so: the chain-entry layout step
(cbs_pack_input), the fused layers and the glue.  The neck layer is a
two-input layer: it reads the upsampled deep feature map and layer 7
straight from their buffers (the channel concatenation happens in its input
loads), so its only glue kernel is the 2x upsample.

With sppf=True the SPPF block follows layer 10: a 1x1 conv, one glue kernel
for its three chained 5x5 max pools (cbs_sppf_pool, writing the three
results side by side along channels), and a 1x1 conv over
concat(conv output, the three pools) as a two-input layer, so the block's
four-way concatenation is never copied.

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
    def __init__(self, prec: str, n: int, seed: int = 0, device="cuda", layout: int | None = None,
                 sppf: bool = False):
        self.prec = prec
        self.n = n
        self.sppf = sppf
        self.device = torch.device(device)
        self.specs = wl.chain_layers(sppf)
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
            if cl.src[0] == "upcat":
                c_in_b = self.specs[cl.src[2]].spec.c_out
            elif cl.src[0] == "sppf":
                c_in_b = 3 * self.specs[cl.src[1]].spec.c_out
            else:
                c_in_b = 0
            desc = make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad, prec=cp,
                             in_layout=self.layout, out_layout=self.layout, c_in_b=c_in_b)
            self.layers.append(FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps,
                                               device=self.device))
        self.outs = [layer.empty_y() for layer in self.layers]
        self.x0 = self.layers[0].empty_x()
        self.neck = next(i for i, cl in enumerate(self.specs) if cl.src[0] == "upcat")
        self.glue = self.layers[self.neck].empty_x()   # upsample2x(deep map): the neck layer's first input
        self.pools = None
        if sppf:
            self.sppf_at = next(i for i, cl in enumerate(self.specs) if cl.src[0] == "sppf")
            self.pools = self.layers[self.sppf_at].empty_x_b()   # the three pooled maps, side by side

    def params(self, i: int, seed: int = 0):
        return wl.layer_params(self.specs[i].spec, seed=seed, layer_index=100 + i)

    def input_of(self, i: int):
        """The device tensor layer i reads (its first input; after its source has run)."""
        src = self.specs[i].src
        if src[0] == "frame":
            return self.x0
        if src[0] in ("layer", "sppf"):
            return self.outs[src[1]]
        return self.glue

    def second_input_of(self, i: int):
        """The second input of a two-input layer, else None."""
        src = self.specs[i].src
        if src[0] == "upcat":
            return self.outs[src[2]]
        return self.pools if src[0] == "sppf" else None

    def launches_per_frame(self) -> int:
        # fused layers, frame packing, one upsample kernel (and one SPPF pool kernel)
        return len(self.layers) + 2 + (1 if self.sppf else 0)

    def _shape(self, a):
        if self.layout == B.CBS_NHWC:
            n, h, w, c = a.shape
        else:
            n, c, h, w = a.shape
        return n, c, h, w

    def glue_before(self, i: int, s: int):
        """Enqueue the glue kernel that layer i's inputs need, if any."""
        src = self.specs[i].src
        if src[0] == "upcat":
            a = self.outs[src[1]]
            n, ca, h, w = self._shape(a)
            B.cbs_upsample2x_concat(a, ca, None, 0, self.glue, n, 2 * h, 2 * w, self.layout, a.element_size(), s)
        elif src[0] == "sppf":
            a = self.outs[src[1]]
            n, c, h, w = self._shape(a)
            B.cbs_sppf_pool(a, self.pools, n, c, h, w, wl.SPPF_POOL_K, self.layout, self.layers[i].prec, s)

    def run(self, frame_nchw: torch.Tensor, stream: int | None = None):
        """One frame batch: pack the frame, then the layers and their glue in order."""
        s = current_stream() if stream is None else stream
        B.cbs_pack_input(self.layers[0].plan, frame_nchw, self.x0, 0.0, s)
        for i, layer in enumerate(self.layers):
            self.glue_before(i, s)
            layer(self.input_of(i), self.outs[i], stream=s, x_b=self.second_input_of(i))
        return self.outs

    def flops(self) -> int:
        return sum(cl.spec.flops(self.n) for cl in self.specs)

    def alg_bytes(self, act_bytes: int) -> int:
        return sum(cl.spec.alg_bytes(self.n, act_bytes) for cl in self.specs)


def to_nchw_numpy(t: torch.Tensor, layout: int) -> np.ndarray:
    a = t.float().cpu().numpy()
    return np.ascontiguousarray(a.transpose(0, 3, 1, 2)) if layout == B.CBS_NHWC else a
