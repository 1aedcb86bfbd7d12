"""Seeded synthetic workloads: layer shapes and input draws.

This module draws random inputs and describes shapes.  It holds none of the
layer's arithmetic, and both the CPU oracle's tests and the GPU path take
their inputs from it.

Distributions (page 1 names the YOLO26N feature-map sizes; the draws stand in
for COCO frames and trained weights, which are not available):
  x ~ N(0, 1); w ~ N(0, 2/fan_in) with fan_in = C_in*k*k (the second argument
  of N is a variance); gamma ~ U(0.5, 1.5); beta, mean ~ N(0, 0.1);
  var ~ U(0.5, 2.0); eps = 1e-3.
Draw order for one layer: x (if the layer draws its own input), w, gamma,
beta, mean, var, all from numpy's PCG64 generator seeded with
seed + 1000 * layer_index, drawn in float64 and rounded to float32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

EPS = 1e-3

# 99.999th percentile of |x| for x ~ N(0, 1): the t with erfc(t / sqrt 2) = 1e-5.
# Per-tensor INT8 activation scale s_x = t / 127 (page 3, "Highlights":
# percentile calibration at the 99.999th percentile).
ABS_NORMAL_P99999 = 4.417173413469
S_X_INT8 = np.float32(ABS_NORMAL_P99999 / 127.0)


@dataclass(frozen=True)
class LayerSpec:
    c_in: int
    c_out: int
    k: int
    stride: int
    h: int           # input height = width
    w: int = 0       # 0: same as h

    @property
    def width(self) -> int:
        return self.w or self.h

    @property
    def pad(self) -> int:
        return self.k // 2

    @property
    def oh(self) -> int:
        return (self.h + 2 * self.pad - self.k) // self.stride + 1

    @property
    def ow(self) -> int:
        return (self.width + 2 * self.pad - self.k) // self.stride + 1

    def flops(self, n: int) -> int:
        """2 * N * C_out * OH * OW * C_in * k^2."""
        return 2 * n * self.c_out * self.oh * self.ow * self.c_in * self.k * self.k

    def alg_bytes(self, n: int, act_bytes: int, w_bytes: int | None = None, extra_per_cout: int = 4) -> int:
        """Input read once + output written once + weights + per-channel vectors."""
        w_bytes = act_bytes if w_bytes is None else w_bytes
        x = n * self.c_in * self.h * self.width * act_bytes
        y = n * self.c_out * self.oh * self.ow * act_bytes
        wt = self.c_out * self.c_in * self.k * self.k * w_bytes
        return x + y + wt + extra_per_cout * self.c_out


# Single fused layer: N=1, 16->32, 3x3, stride 1, pad 1, 40x40 (OW = 40 is not
# a multiple of 16, the width at which page 1's padded-row-stride bug bit).
SINGLE_LAYER = LayerSpec(16, 32, 3, 1, 40)

# The twelve-layer list of YOLO26n-scale shapes (C_in, C_out, k, stride, H=W).
LAYER_LIST = (
    LayerSpec(3, 16, 3, 2, 640),
    LayerSpec(16, 32, 3, 2, 320),
    LayerSpec(32, 32, 1, 1, 160),
    LayerSpec(32, 64, 3, 2, 160),
    LayerSpec(64, 64, 1, 1, 80),
    LayerSpec(64, 64, 3, 1, 80),
    LayerSpec(64, 128, 3, 2, 80),
    LayerSpec(128, 128, 3, 1, 40),
    LayerSpec(128, 256, 3, 2, 40),
    LayerSpec(256, 256, 1, 1, 20),
    LayerSpec(256, 256, 3, 1, 20),
    LayerSpec(384, 128, 1, 1, 40),
)


@dataclass(frozen=True)
class ChainLayer:
    spec: LayerSpec
    src: tuple   # ("frame",) | ("layer", i) | ("upcat", i_upsampled, i_skip) | ("sppf", i)


def _repeats(c: int, size: int, count: int):
    return [LayerSpec(c, c, 1 if i % 2 == 0 else 3, 1, size) for i in range(count)]


def chain_layers(sppf: bool = False) -> tuple:
    """The 40-layer whole-frame chain, or with sppf=True the whole synthetic
    frame: the same chain with the SPPF block of the detector's backbone
    inserted after layer 10.

    Layers 0..10: the list's first eleven layers in order, from the frame.
    Layer 11: the list's 384->128 1x1 layer on concat(upsample2x(out10), out7)
    (neck glue: 256 channels at 20x20 upsampled to 40x40 plus 128 at 40x40).
    Then 28 stride-1 repeats alternating 1x1 and 3x3 (starting with 1x1):
    10 at 80x80 with 64 channels branching from layer 5, 9 at 40x40 with 128
    channels following layer 11, 9 at 20x20 with 256 channels branching from
    layer 10.

    With sppf=True (42 layers), layer 11 is the SPPF's first 1x1 conv
    (256->128 at 20x20, on out10), its output goes through three chained 5x5
    stride-1 max pools, and layer 12 is the SPPF's second 1x1 conv (512->256)
    on concat(out11, pool(out11), pool^2(out11), pool^3(out11)) (source
    ("sppf", 11)).  Layer 13 is the neck layer on concat(upsample2x(out12),
    out7), and the 20x20 repeats branch from the SPPF output (layer 12); the
    80x80 repeats still branch from layer 5 and the 40x40 ones follow the
    neck layer.
    """
    out = []
    for i, spec in enumerate(LAYER_LIST[:11]):
        out.append(ChainLayer(spec, ("frame",) if i == 0 else ("layer", i - 1)))
    deep = 10
    if sppf:
        out.append(ChainLayer(LayerSpec(256, 128, 1, 1, 20), ("layer", 10)))
        out.append(ChainLayer(LayerSpec(512, 256, 1, 1, 20), ("sppf", 11)))
        deep = 12
    neck = len(out)
    out.append(ChainLayer(LAYER_LIST[11], ("upcat", deep, 7)))
    for stage_c, size, count, first_src in ((64, 80, 10, 5), (128, 40, 9, neck), (256, 20, 9, deep)):
        for j, spec in enumerate(_repeats(stage_c, size, count)):
            src = ("layer", first_src) if j == 0 else ("layer", len(out) - 1)
            out.append(ChainLayer(spec, src))
    assert len(out) == (42 if sppf else 40)
    return tuple(out)


# Max pool of the SPPF block: 5x5, stride 1, padding 2.
SPPF_POOL_K = 5


@dataclass
class LayerParams:
    w: np.ndarray      # [C_out, C_in, k, k] float32
    gamma: np.ndarray  # [C_out] float32
    beta: np.ndarray
    mean: np.ndarray
    var: np.ndarray
    eps: float = EPS


def _rng(seed: int, layer_index: int):
    return np.random.default_rng(seed + 1000 * layer_index)


def _draw_params(rng, spec: LayerSpec) -> LayerParams:
    fan_in = spec.c_in * spec.k * spec.k
    w = rng.normal(0.0, np.sqrt(2.0 / fan_in), size=(spec.c_out, spec.c_in, spec.k, spec.k))
    gamma = rng.uniform(0.5, 1.5, size=spec.c_out)
    beta = rng.normal(0.0, np.sqrt(0.1), size=spec.c_out)
    mean = rng.normal(0.0, np.sqrt(0.1), size=spec.c_out)
    var = rng.uniform(0.5, 2.0, size=spec.c_out)
    f = lambda a: np.ascontiguousarray(a, dtype=np.float32)  # noqa: E731
    return LayerParams(f(w), f(gamma), f(beta), f(mean), f(var))


def layer_inputs(spec: LayerSpec, n: int, seed: int = 0, layer_index: int = 0):
    """(x [n, C_in, H, W] float32, LayerParams) for an independent layer."""
    rng = _rng(seed, layer_index)
    x = np.ascontiguousarray(rng.standard_normal(size=(n, spec.c_in, spec.h, spec.width)), dtype=np.float32)
    return x, _draw_params(rng, spec)


def layer_params(spec: LayerSpec, seed: int = 0, layer_index: int = 0) -> LayerParams:
    """Parameters of a layer whose input comes from another layer (chain)."""
    rng = _rng(seed, layer_index)
    return _draw_params(rng, spec)


def frame(n: int, seed: int = 0, size: int = 640) -> np.ndarray:
    """Chain input: [n, 3, size, size] float32 ~ N(0, 1) (seed offset 999)."""
    rng = np.random.default_rng(seed + 999)
    return np.ascontiguousarray(rng.standard_normal(size=(n, 3, size, size)), dtype=np.float32)
