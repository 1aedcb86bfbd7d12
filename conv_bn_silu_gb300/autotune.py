"""Measure candidate plans per layer shape on the GPU and write the table
that `tuning.tuned_desc` reads.

For every distinct layer shape of the benchmark workloads (the twelve-layer
list at batch 16 in BF16, TF32 and INT8, the 40-layer chain at batch 16 in
BF16, TF32 and INT8, both at batch 1 in FP32, and the list at batches 1 and 16 in
FP32 with NHWC activations on the 3xTF32 kernel), each candidate configuration is
planned, folded and timed as a CUDA graph of repeated launches over rotating
input copies.  A shape gets a table entry when its fastest candidate beats the
cost-model plan by 3% or more.

    python -m conv_bn_silu_gb300.autotune OUT.json [--reps 10]

One shape under given force fields, timed the same way (no table written):

    python -m conv_bn_silu_gb300.autotune --time PREC N C_IN C_OUT K STRIDE H W \
        [--force FIELD=VALUE ...] [--reps 10]
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import time

import torch

from . import _binding as B
from . import workloads as wl
from .layer import FusedConvBnSilu, make_desc
from .tuning import FORCE_FIELDS, shape_key

PRECS = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16, "int8": B.CBS_INT8}
SIMT_TILES = ((128, 128), (128, 64), (64, 64), (128, 32), (256, 16), (64, 128))


def workload_shapes():
    """(precision, batch, LayerSpec, layout) of every layer the benchmarks run."""
    out = []
    chain = [cl.spec for cl in wl.chain_layers()]
    for prec in ("bf16", "tf32", "int8"):
        out += [(prec, 16, s, B.CBS_NHWC) for s in wl.LAYER_LIST]
    for prec in ("bf16", "tf32", "int8"):
        out += [(prec, 16, s, B.CBS_NHWC) for s in chain]
    out += [("fp32", 1, s, B.CBS_NCHW) for s in list(wl.LAYER_LIST) + chain + [wl.SINGLE_LAYER]]
    # FP32 with NHWC activations: the 3xTF32 tensor-core kernel
    out += [("fp32", n, s, B.CBS_NHWC) for n in (16, 1) for s in wl.LAYER_LIST]
    seen, uniq = set(), []
    for prec, n, s, lay in out:
        k = (prec, n, s, lay)
        if k not in seen:
            seen.add(k)
            uniq.append(k)
    return uniq


def candidates(prec, spec, base):
    """Descriptor force-field sets to try for one shape."""
    full = min(256, -(-spec.c_out // 16) * 16)
    bns = [b for b in (32, 48, 64, 96, 128, 192, 256) if b <= full] or [full]
    if prec == "fp32":
        if base.in_layout == B.CBS_NHWC:
            # 3xTF32: N tile and K parts; the variant is forced with them (a
            # forced tile field alone keeps an FP32 plan on the CUDA cores).
            for sk, bn in itertools.product((1, 2, 3, 4, 5, 6, 8, 9, 12, 16), bns):
                yield dict(force_variant=B.CBS_VARIANT_TC_TF32X3, force_split_k=sk, force_block_n=bn)
        else:
            # the CUDA-core kernel
            for (bm, bn), sk in itertools.product(SIMT_TILES, (1, 2, 3, 4, 6, 8, 12, 16)):
                yield dict(force_variant=B.CBS_VARIANT_SIMT_FP32, force_block_m=bm, force_block_n=bn,
                           force_split_k=sk)
            # 3xTF32 reading the NCHW input: the converter warps' own loads,
            # and flat TMA boxes where every filter row of a tile is one
            # aligned run of a channel row
            if spec.c_in % 8 == 0:
                flat = (spec.stride == 1 and spec.k <= 7 and spec.width % 4 == 0 and
                        (base.n == 1 or (spec.oh * spec.ow) % 128 == 0))
                for sk, bn in itertools.product((1, 2, 3, 4, 5, 6, 8), bns):
                    yield dict(force_variant=B.CBS_VARIANT_TC_TF32X3, force_split_k=sk, force_block_n=bn)
                    if flat:
                        yield dict(force_variant=B.CBS_VARIANT_TC_TF32X3, force_split_k=sk, force_block_n=bn,
                                   force_window=1)
    elif prec == "int8":
        for kg, bn in itertools.product((1, 2, 3, 4), bns):
            yield dict(force_k_group=kg, force_block_n=bn)
    else:
        for bm, kg, br, bn in itertools.product((128, 256), (1, 2, 3, 4), (-1, 1), bns):
            yield dict(force_block_m=bm, force_k_group=kg, force_b_resident=br, force_block_n=bn,
                       force_issuer_split=-1)
            if bm == 128 and bn <= 128:
                # 128-pixel tiles: K stages alternating between the two MMA issuers
                yield dict(force_block_m=bm, force_k_group=kg, force_b_resident=br, force_block_n=bn,
                           force_issuer_split=1)
        if spec.stride == 1 or (spec.stride == 2 and spec.k == 3):
            for bm, br, bn in itertools.product((128, 256), (-1, 1), bns):
                yield dict(force_block_m=bm, force_b_resident=br, force_block_n=bn, force_window=1)


class Timer:
    def __init__(self, reps):
        self.reps = reps
        self.stream = torch.cuda.Stream()

    def __call__(self, layer, xs, ys, s_y):
        st = self.stream
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            layer(xs[0], ys[0], s_y=s_y, stream=st.cuda_stream)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=st):
                for r in range(self.reps):
                    layer(xs[r % len(xs)], ys[r % len(ys)], s_y=s_y, stream=st.cuda_stream)
            torch.cuda.synchronize()
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            g.replay()
            e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / self.reps


def tune(reps: int = 10, log=print):
    timer = Timer(reps)
    plans = {}
    t_start = time.time()
    for prec, n, spec, lay in workload_shapes():
        cp = PRECS[prec]
        base = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad, prec=cp,
                         in_layout=lay, out_layout=lay)
        auto_plan = B.cbs_plan(base)
        if auto_plan.variant == B.CBS_VARIANT_STEM:
            continue
        x, p = wl.layer_inputs(spec, n, layer_index=0)
        s_x = float(wl.S_X_INT8) if prec == "int8" else 0.0
        auto = FusedConvBnSilu(base, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x, tuned=False)
        xd = torch.from_numpy(x).cuda()
        x0 = auto.pack_input(xd) if (prec != "fp32" or lay == B.CBS_NHWC) else xd
        nbytes = x0.numel() * x0.element_size()
        copies = int(min(8, max(2, math.ceil((256 << 20) / max(nbytes, 1)))))
        xs = [x0] + [x0.clone() for _ in range(copies - 1)]
        ys = [auto.empty_y() for _ in range(copies)]
        s_y = 0.05
        t_auto = timer(auto, xs, ys, s_y)
        best_t, best_f, best_desc = t_auto, None, None
        tried = 0
        for force in candidates(prec, spec, base):
            d = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad, prec=cp,
                          in_layout=lay, out_layout=lay, **force)
            try:
                pl = B.cbs_plan(d)
            except B.CbsError:
                continue
            if "force_block_n" in force and pl.block_n != force["force_block_n"]:
                continue
            layer = FusedConvBnSilu(d, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x, tuned=False)
            t = timer(layer, xs, [layer.empty_y() for _ in range(copies)], s_y)
            tried += 1
            if t < best_t:
                best_t, best_f, best_desc = t, force, pl
        key = shape_key(base)
        note = f"{prec} n{n} {spec.c_in}->{spec.c_out} k{spec.k} s{spec.stride} {spec.h}x{spec.width}"
        if best_f is not None and best_t < 0.97 * t_auto:
            plans[key] = {"force": {k: int(v) for k, v in best_f.items() if k in FORCE_FIELDS},
                          "us": round(best_t, 2), "auto_us": round(t_auto, 2), "layer": note,
                          "plan": f"bm{best_desc.block_m} bn{best_desc.block_n} kg{best_desc.k_group} "
                                  f"br{best_desc.b_resident} win{best_desc.window} split{best_desc.split_k}"}
            log(f"{note}: {t_auto:.1f} -> {best_t:.1f} us ({plans[key]['plan']}, {tried} tried)")
        else:
            log(f"{note}: {t_auto:.1f} us, cost-model plan kept ({tried} tried)")
        del xs, ys
        torch.cuda.empty_cache()
    status = B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream)
    if status != B.CBS_OK:
        raise RuntimeError(f"a kernel reported {B.status_name(status)} while tuning")
    log(f"tuned {len(plans)} shapes in {time.time() - t_start:.0f} s")
    return plans


def time_plan(prec: str, n: int, spec: wl.LayerSpec, force: dict, reps: int = 10):
    """Microseconds per launch of one layer shape planned with `force` (NHWC
    for the tensor-core precisions, NCHW for FP32), and its plan."""
    cp = PRECS[prec]
    lay = B.CBS_NCHW if prec == "fp32" else B.CBS_NHWC
    d = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad, prec=cp,
                  in_layout=lay, out_layout=lay, **force)
    x, p = wl.layer_inputs(spec, n, layer_index=0)
    s_x = float(wl.S_X_INT8) if prec == "int8" else 0.0
    layer = FusedConvBnSilu(d, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x, tuned=False)
    xd = torch.from_numpy(x).cuda()
    x0 = layer.pack_input(xd) if (prec != "fp32" or lay == B.CBS_NHWC) else xd
    nbytes = x0.numel() * x0.element_size()
    copies = int(min(8, max(2, math.ceil((256 << 20) / max(nbytes, 1)))))
    xs = [x0] + [x0.clone() for _ in range(copies - 1)]
    ys = [layer.empty_y() for _ in range(copies)]
    us = Timer(reps)(layer, xs, ys, 0.05)
    status = B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream)
    if status != B.CBS_OK:
        raise RuntimeError(f"a kernel reported {B.status_name(status)}")
    return us, layer.plan


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("out", nargs="?")
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--time", nargs=8, metavar=("PREC", "N", "C_IN", "C_OUT", "K", "STRIDE", "H", "W"))
    ap.add_argument("--force", action="append", default=[], metavar="FIELD=VALUE")
    args = ap.parse_args()
    if args.time:
        prec = args.time[0]
        n, c_in, c_out, k, stride, h, w = (int(v) for v in args.time[1:])
        force = {}
        for f in args.force:
            name, _, v = f.partition("=")
            if name not in FORCE_FIELDS:
                raise SystemExit(f"unknown force field {name} (one of {', '.join(FORCE_FIELDS)})")
            force[name] = int(v)
        us, pl = time_plan(prec, n, wl.LayerSpec(c_in, c_out, k, stride, h, w), force, args.reps)
        print(f"{prec} n{n} {c_in}->{c_out} k{k} s{stride} {h}x{w} {force}: {us:.2f} us "
              f"(bm{pl.block_m} bn{pl.block_n} kg{pl.k_group} st{pl.stages} br{pl.b_resident} win{pl.window} "
              f"split{pl.split_k} iss{pl.issuer_split})")
        return
    if not args.out:
        ap.error("OUT.json is required unless --time is given")
    plans = tune(args.reps)
    meta = {"device": torch.cuda.get_device_name(0), "created_by": "conv_bn_silu_gb300/autotune.py",
            "timing": f"CUDA graph of {args.reps} launches over rotating input copies, second replay timed",
            "plans": plans}
    with open(args.out, "w") as f:
        json.dump(meta, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
