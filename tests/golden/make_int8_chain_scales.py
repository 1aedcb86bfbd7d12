"""Write tests/golden/int8_chain_scales.json: the INT8 output scale of each
layer of the 40-layer chain.

s_y[i] = p99.999(|y_i|) / 127, nearest rank, over the CPU oracle's FP32
output of chain layer i for the seeded synthetic frame at batch 1 (page 3,
"Highlights": percentile calibration at the 99.999th percentile).  The two
layers whose outputs the neck layer concatenates (the upsampled layer 10 and
layer 7) share one scale, the larger of the two, because the INT8 layer reads
both inputs with one scale.  Calls only the oracle and the input generator
(the neck's 2x upsample and concatenation are copies, done here with numpy).
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
    specs = wl.chain_layers()
    frame = wl.frame(1)
    outs, scales = [], []
    for i, cl in enumerate(specs):
        s, src = cl.spec, cl.src
        if src[0] == "frame":
            x = frame
        elif src[0] == "layer":
            x = outs[src[1]]
        else:
            a = outs[src[1]]
            x = np.concatenate([a.repeat(2, axis=2).repeat(2, axis=3), outs[src[2]]], axis=1)
        p = wl.layer_params(s, seed=0, layer_index=100 + i)
        y = oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad)
        outs.append(y)
        scales.append(p99999_over_127(y))
    for cl in specs:
        if cl.src[0] == "upcat":
            a, b = cl.src[1], cl.src[2]
            scales[a] = scales[b] = max(scales[a], scales[b])
    out = {"source": "p99.999(|y|)/127, nearest rank, oracle FP32 chain output, batch 1, seed 0; "
                     "the neck's two inputs share the larger scale",
           "input_scale": float(wl.S_X_INT8), "chain": scales}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "int8_chain_scales.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()
