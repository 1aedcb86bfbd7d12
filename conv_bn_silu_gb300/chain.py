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

prec="int8" runs the chain on INT8 layers (page 3, "Edge optimisation of
YOLO26": per-channel weight scales, per-tensor activation scales).  Each
layer's output scale comes from a calibration table (`out_scales`); a layer
reads its input with the scale of the layer that wrote it (the frame: the
input scale).  `keep_float` names layers that run in float instead (BF16 by
default, or FP32), as page 3's layer-sensitivity analysis keeps its most
sensitive layers in float.  Where a layer's input format differs from its
source's output format a seam kernel converts it: cbs_dequantize_i8 (codes
to float with the source's scale) or cbs_quantize_i8 (float to codes with
the source's calibrated scale).  Seams are made once per (source, format)
and shared by that source's consumers.

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

PRECS = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16, "int8": B.CBS_INT8}


class Chain:
    def __init__(self, prec: str, n: int, seed: int = 0, device="cuda", layout: int | None = None,
                 sppf: bool = False, out_scales=None, in_scale: float | None = None, keep_float=(),
                 float_prec: str = "bf16"):
        self.prec = prec
        self.n = n
        self.sppf = sppf
        self.device = torch.device(device)
        self.specs = wl.chain_layers(sppf)
        if layout is None:
            layout = B.CBS_NCHW if prec == "fp32" else B.CBS_NHWC
        if prec != "fp32" and layout != B.CBS_NHWC:
            raise ValueError("the tensor-core precisions run the chain in NHWC")
        self.layout = layout
        self.keep_float = frozenset(int(i) for i in keep_float)
        if prec == "int8":
            if sppf:
                raise ValueError("the INT8 chain runs without the SPPF block")
            if out_scales is None or len(out_scales) != len(self.specs):
                raise ValueError("the INT8 chain needs one calibrated output scale per layer")
            if float_prec not in ("bf16", "fp32"):
                raise ValueError("layers kept in float run in BF16 or FP32")
            for cl in self.specs:
                if cl.src[0] == "upcat" and out_scales[cl.src[1]] != out_scales[cl.src[2]]:
                    raise ValueError("the two inputs of a two-input layer need one scale")
        elif self.keep_float:
            raise ValueError("keep_float applies to the INT8 chain")
        self.out_scales = None if out_scales is None else [float(v) for v in out_scales]
        self.in_scale = float(wl.S_X_INT8 if in_scale is None else in_scale)
        # Precision each layer runs in.
        self.layer_prec = [(float_prec if i in self.keep_float else "int8") if prec == "int8" else prec
                           for i in range(len(self.specs))]
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
            lp = self.layer_prec[i]
            desc = make_desc(n, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad, prec=PRECS[lp],
                             in_layout=self.layout, out_layout=self.layout, c_in_b=c_in_b)
            s_x = self.input_scale(i) if lp == "int8" else 0.0
            self.layers.append(FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x,
                                               device=self.device))
        self.outs = [layer.empty_y() for layer in self.layers]
        self.x0 = self.layers[0].empty_x()
        self.neck = next(i for i, cl in enumerate(self.specs) if cl.src[0] == "upcat")
        self.glue = self.layers[self.neck].empty_x()   # upsample2x(deep map): the neck layer's first input
        self.pools = None
        if sppf:
            self.sppf_at = next(i for i, cl in enumerate(self.specs) if cl.src[0] == "sppf")
            self.pools = self.layers[self.sppf_at].empty_x_b()   # the three pooled maps, side by side
        # Seam buffers: (source layer, element type) -> the source's output in that type.
        self.seams = {}
        for i, cl in enumerate(self.specs):
            for j in self.sources(i):
                want = self.layers[i].x_dtype
                if self.outs[j].dtype != want and (j, want) not in self.seams:
                    self.seams[(j, want)] = torch.empty(self.outs[j].shape, dtype=want, device=self.device)

    def sources(self, i: int):
        """Layers whose outputs layer i reads (in input order)."""
        src = self.specs[i].src
        if src[0] in ("layer", "sppf"):
            return [src[1]]
        if src[0] == "upcat":
            return [src[1], src[2]]
        return []

    def input_scale(self, i: int) -> float:
        """Scale of layer i's INT8 input codes: the scale of the layer that
        wrote them (for the frame, the input scale)."""
        src = self.specs[i].src
        return self.in_scale if src[0] == "frame" else self.out_scales[src[1]]

    def out_of(self, j: int, dtype):
        """Layer j's output in `dtype` (the seam buffer when the types differ)."""
        return self.outs[j] if self.outs[j].dtype == dtype else self.seams[(j, dtype)]

    def convert_seams(self, i: int, s: int):
        """Enqueue the seam conversions layer i's inputs need (each seam once per
        step, at its first consumer)."""
        want = self.layers[i].x_dtype
        for j in self.sources(i):
            if self.outs[j].dtype == want or self._first_consumer.get((j, want)) != i:
                continue
            src = self.outs[j]
            if want == torch.int8:
                fp = B.CBS_BF16 if src.dtype == torch.bfloat16 else B.CBS_FP32
                B.cbs_quantize_i8(src, fp, self.seams[(j, want)], src.numel(), self.out_scales[j], 0, s)
            else:
                fp = B.CBS_BF16 if want == torch.bfloat16 else B.CBS_FP32
                B.cbs_dequantize_i8(src, self.seams[(j, want)], src.numel(), self.out_scales[j], 0, fp, s)

    @property
    def _first_consumer(self):
        if not hasattr(self, "_fc"):
            self._fc = {}
            for i in range(len(self.specs)):
                for j in self.sources(i):
                    key = (j, self.layers[i].x_dtype)
                    self._fc.setdefault(key, i)
        return self._fc

    def params(self, i: int, seed: int = 0):
        return wl.layer_params(self.specs[i].spec, seed=seed, layer_index=100 + i)

    def input_of(self, i: int):
        """The device tensor layer i reads (its first input; after its source has run)."""
        src = self.specs[i].src
        if src[0] == "frame":
            return self.x0
        if src[0] in ("layer", "sppf"):
            return self.out_of(src[1], self.layers[i].x_dtype)
        return self.glue

    def second_input_of(self, i: int):
        """The second input of a two-input layer, else None."""
        src = self.specs[i].src
        if src[0] == "upcat":
            return self.out_of(src[2], self.layers[i].x_dtype)
        return self.pools if src[0] == "sppf" else None

    def launches_per_frame(self) -> int:
        # fused layers, frame packing, one upsample kernel, the SPPF pool kernel, the seams
        return len(self.layers) + 2 + (1 if self.sppf else 0) + len(self.seams)

    def _shape(self, a):
        if self.layout == B.CBS_NHWC:
            n, h, w, c = a.shape
        else:
            n, c, h, w = a.shape
        return n, c, h, w

    def glue_before(self, i: int, s: int):
        """Enqueue the seam conversions and the glue kernel that layer i's
        inputs need, if any."""
        self.convert_seams(i, s)
        src = self.specs[i].src
        if src[0] == "upcat":
            a = self.out_of(src[1], self.layers[i].x_dtype)
            n, ca, h, w = self._shape(a)
            B.cbs_upsample2x_concat(a, ca, None, 0, self.glue, n, 2 * h, 2 * w, self.layout, a.element_size(), s)
        elif src[0] == "sppf":
            a = self.outs[src[1]]
            n, c, h, w = self._shape(a)
            B.cbs_sppf_pool(a, self.pools, n, c, h, w, wl.SPPF_POOL_K, self.layout, self.layers[i].prec, s)

    def pack_frame(self, frame_nchw: torch.Tensor, s: int):
        """The chain-entry layout step (and, for an INT8 first layer, the input quantiser)."""
        s_x = self.in_scale if self.layer_prec[0] == "int8" else 0.0
        B.cbs_pack_input(self.layers[0].plan, frame_nchw, self.x0, s_x, s)

    def call(self, i: int, s: int):
        """Enqueue layer i (after glue_before(i))."""
        layer = self.layers[i]
        s_y = self.out_scales[i] if self.layer_prec[i] == "int8" else None
        layer(self.input_of(i), self.outs[i], s_y=s_y, stream=s, x_b=self.second_input_of(i))

    def run(self, frame_nchw: torch.Tensor, stream: int | None = None):
        """One frame batch: pack the frame, then the layers and their glue in order."""
        s = current_stream() if stream is None else stream
        self.pack_frame(frame_nchw, s)
        for i in range(len(self.layers)):
            self.glue_before(i, s)
            self.call(i, s)
        return self.outs

    def flops(self) -> int:
        return sum(cl.spec.flops(self.n) for cl in self.specs)

    def alg_bytes(self, act_bytes: int | None = None) -> int:
        """Algorithmic bytes of one frame batch; act_bytes None: each layer's own
        element size (an INT8 chain with layers kept in float)."""
        return sum(cl.spec.alg_bytes(self.n, act_bytes or self.layers[i].empty_y().element_size())
                   for i, cl in enumerate(self.specs))


def to_nchw_numpy(t: torch.Tensor, layout: int) -> np.ndarray:
    a = t.float().cpu().numpy()
    return np.ascontiguousarray(a.transpose(0, 3, 1, 2)) if layout == B.CBS_NHWC else a
