"""Write tests/golden/int8_scales.json: the INT8 output scale of each list layer.

s_y = p99.999(|y|) / 127, nearest rank, over the CPU oracle's FP32 output of
the layer at batch 1 on the seeded synthetic input (page 3, "Highlights":
percentile calibration at the 99.999th percentile).  Calls only the oracle
and the input generator.
"""
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from conv_bn_silu_gb300 import workloads as wl  # noqa: E402


def p99999_over_127(y):
    a = np.sort(np.abs(np.asarray(y, np.float64)).ravel())
    rank = math.ceil(0.99999 * a.size)
    return float(np.float32(a[rank - 1] / 127.0))


def main():
    out = {"source": "p99.999(|y|)/127, nearest rank, oracle FP32 output, batch 1, seed 0",
           "layer_list": []}
    for i, s in enumerate(wl.LAYER_LIST):
        x, p = wl.layer_inputs(s, 1, seed=0, layer_index=i)
        y = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad)
        out["layer_list"].append(p99999_over_127(y))
    x, p = wl.layer_inputs(wl.SINGLE_LAYER, 1)
    s = wl.SINGLE_LAYER
    out["single_layer"] = p99999_over_127(
        oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "int8_scales.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()
