"""Benchmark of the fused Conv2d + folded BN + SiLU layer on GB300.

Default workload: the twelve-layer YOLO26n-scale list at batch 1 in FP32
(CUDA-core variant), NCHW in and out.  One step = the twelve fused layers,
each on its own seeded synthetic input, all resident in HBM.  The K timed
steps run as one captured CUDA graph (no host launch overhead inside the
timed region) with timing events between every kernel, so each launch's
device duration is measured in the same run.  Inputs and outputs rotate over
five copies (5 x 55 MB > the 126 MB L2), so no step finds its inputs in L2
from the step before.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores on the same workload and metric instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from conv_bn_silu_gb300 import workloads as wl  # noqa: E402

# FP32 CUDA-core peak: 152 SMs x 128 FP32 lanes x 2 FLOP per FMA x 2.07 GHz.
SM_COUNT, FP32_LANES, SM_MAX_GHZ = 152, 128, 2.070
FP32_ALU_PEAK_TFLOPS = SM_COUNT * FP32_LANES * 2 * SM_MAX_GHZ / 1e3
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 2**20


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- workloads
WORKLOADS = {
    "layer_list_fp32_n1": dict(layers=wl.LAYER_LIST, n=1, prec="fp32"),
    "single_layer_fp32_n1": dict(layers=(wl.SINGLE_LAYER,), n=1, prec="fp32"),
}


def act_bytes(prec: str) -> int:
    return {"fp32": 4, "tf32": 4, "bf16": 2, "int8": 1}[prec]


def build_layers(name: str, device):
    import torch
    from conv_bn_silu_gb300 import _binding as B
    from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
    cfg = WORKLOADS[name]
    prec = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16, "int8": B.CBS_INT8}[cfg["prec"]]
    layers = []
    for i, spec in enumerate(cfg["layers"]):
        x, p = wl.layer_inputs(spec, cfg["n"], seed=0, layer_index=i)
        desc = make_desc(cfg["n"], spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                         prec=prec)
        layer = FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, device=device)
        layers.append((spec, layer, x))
    return cfg, layers


def run_ours(args, rank: int, world: int):
    import torch
    from conv_bn_silu_gb300 import _binding as B

    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(device)
    cfg, layers = build_layers(args.workload, device)
    n = cfg["n"]
    peaks, peak_src = load_peaks()
    ab = act_bytes(cfg["prec"])

    # Resident inputs/outputs, rotated over R copies so the working set per
    # rotation exceeds L2.
    step_bytes = sum(s.alg_bytes(n, ab) for s, _, _ in layers)
    R = max(2, int(np.ceil(2 * L2_BYTES / step_bytes)) + 1)
    xs = [[torch.from_numpy(x).to(device) for (_, _, x) in layers] for _ in range(R)]
    ys = [[layer.empty_y() for (_, layer, _) in layers] for _ in range(R)]
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device)
    sid = stream.cuda_stream

    def step(r, events=None):
        for j, (_, layer, _) in enumerate(layers):
            if events is not None:
                events[j].record(stream)
            layer(xs[r][j], ys[r][j], stream=sid)
        if events is not None:
            events[len(layers)].record(stream)

    # Warm-up: W steps, eager.
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i % R)
    torch.cuda.synchronize()

    # Capture exactly K steps (with an event between every launch) in one graph.
    K = args.steps
    nl = len(layers)
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(nl + 1)] for _ in range(K)]
    except TypeError:  # older torch without external events
        evs = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(K):
                step(i % R, evs[i] if evs is not None else None)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph.replay()  # one untimed replay of the instantiated graph
    torch.cuda.synchronize()

    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(device.index)
    time.sleep(0.3)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        graph.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    # Per-launch durations: read the in-graph events of the timed replay now.
    per_layer_us = None
    if evs is not None:
        per_layer_us = np.zeros(len(layers))
        for i in range(args.steps):
            for j in range(len(layers)):
                per_layer_us[j] += evs[i][j].elapsed_time(evs[i][j + 1]) * 1e3
        per_layer_us /= args.steps
    if world > 1:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)
    # keep the GPU busy with the same workload for >= 1 s so the clock sampler
    # sees this load (the timed region itself may be shorter than a sample)
    tend = time.time() + 1.0
    while time.time() < tend:
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
    clocks = sampler.stop()

    ms_step = total_ms / K
    if world > 1:
        t = torch.tensor([ms_step], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_step = float(t.item())


    flops_step = sum(s.flops(n) for s, _, _ in layers)
    value = flops_step * world / (ms_step * 1e-3) / 1e12

    # Roofline of the dominant kernel (the FP32 CUDA-core conv kernel: every
    # launch of this workload) and per layer.
    hbm = float(peaks["hbm_gbs"])
    layer_rows = []
    for j, (s, layer, _) in enumerate(layers):
        f, by = s.flops(n), s.alg_bytes(n, ab)
        t_roof_us = max(f / (FP32_ALU_PEAK_TFLOPS * 1e12), by / (hbm * 1e9)) * 1e6
        row = {"layer": j + 1, "shape": f"{s.c_in}->{s.c_out} k{s.k} s{s.stride} {s.h}",
               "tile": f"{layer.plan.block_m}x{layer.plan.block_n}", "split_k": layer.plan.split_k,
               "mflop": round(f / 1e6, 2), "alg_mb": round(by / 1e6, 3), "roofline_us": round(t_roof_us, 3)}
        if per_layer_us is not None:
            row["us"] = round(float(per_layer_us[j]), 3)
            row["tflops"] = round(f / (per_layer_us[j] * 1e-6) / 1e12, 3)
            row["frac_of_roofline"] = round(t_roof_us / per_layer_us[j], 4)
        layer_rows.append(row)
    if per_layer_us is not None:
        kern_us = float(per_layer_us.sum())
    else:
        kern_us = ms_step * 1e3
    achieved = flops_step / (kern_us * 1e-6) / 1e12
    roofline = {"bound": "alu", "kernel": "simt_conv_kernel (FP32 FMA, all launches)",
                "achieved": round(achieved, 3), "peak": round(FP32_ALU_PEAK_TFLOPS, 2), "unit": "TFLOP/s",
                "frac": round(achieved / FP32_ALU_PEAK_TFLOPS, 4),
                "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz",
                "traffic": None,
                "sum_layer_roofline_us": round(sum(r["roofline_us"] for r in layer_rows), 2),
                "frac_of_layer_roofline_sum": (round(sum(r["roofline_us"] for r in layer_rows) / kern_us, 4)
                                               if kern_us > 0 else None)}

    e2e = run_e2e(layers, n, device, stream, args, flops_step, world)
    out = {
        "metric": "fused conv+BN+SiLU TFLOP/s & us/frame over the layer list; % of roofline",
        "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "us_per_frame": round(ms_step * 1e3 / n, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded N(0,1) inputs, He-init weights, random BN statistics)",
        "config": {"workload": args.workload, "layers": len(layers), "batch": n, "layout": "NCHW",
                   "l2": f"inputs larger than L2: {R} rotating copies of the step's {step_bytes / 1e6:.1f} MB",
                   "timing": "K steps captured in one CUDA graph, events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline, "layers": layer_rows,
        "gpu_launches": K * len(layers),
        "e2e": e2e, "clocks": clocks, "peaks_source": peak_src,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, layers)
    return out


def run_e2e(layers, n, device, stream, args, flops_step, world):
    """Same metric through the public API with host buffers: each step copies
    its inputs from pinned host memory, runs the layers and reads every
    output back; the host waits for the result."""
    import torch
    xs_h = [torch.from_numpy(x).pin_memory() for (_, _, x) in layers]
    ys_h = [torch.empty(layer.y_shape(), dtype=layer.x_dtype).pin_memory() for (_, layer, _) in layers]
    xs_d = [torch.empty_like(x, device=device) for x in xs_h]
    ys_d = [layer.empty_y() for (_, layer, _) in layers]
    sid = stream.cuda_stream
    steps = max(3, min(args.steps, 50))

    def one():
        with torch.cuda.stream(stream):
            for j, (_, layer, _) in enumerate(layers):
                xs_d[j].copy_(xs_h[j], non_blocking=True)
                layer(xs_d[j], ys_d[j], stream=sid)
                ys_h[j].copy_(ys_d[j], non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        one()
    t = time.perf_counter()
    for _ in range(steps):
        one()
    dt = (time.perf_counter() - t) / steps
    h2d = sum(x.numel() * x.element_size() for x in xs_h)
    d2h = sum(y.numel() * y.element_size() for y in ys_h)
    return {"value": round(flops_step * world / dt / 1e12, 4), "unit": "TFLOP/s",
            "ms_per_step": round(dt * 1e3, 4), "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def cpu_baseline(cfg, layers, budget_s: float = 20.0):
    """The CPU oracle as it stands, on the host cores, on a bounded sample of
    the same workload: layers of the list in order until the budget is
    spent (the last one included)."""
    import oracle
    done_flops, t0, used = 0, time.perf_counter(), []
    for i, (spec, _, x) in enumerate(layers):
        _, p = wl.layer_inputs(spec, cfg["n"], seed=0, layer_index=i)
        oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad)
        done_flops += spec.flops(cfg["n"])
        used.append(i + 1)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done_flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"layers {used[0]}..{used[-1]} of the list at batch {cfg['n']}, one pass, double arithmetic"}


def run_reference(args, rank: int, world: int):
    """The oracle on the host cores: each step is one layer of the list
    (round robin), full size."""
    if rank != 0:
        return None
    import oracle
    cfg = WORKLOADS[args.workload]
    specs = cfg["layers"]
    inputs = [wl.layer_inputs(s, cfg["n"], seed=0, layer_index=i) for i, s in enumerate(specs)]

    def step(i):
        j = i % len(specs)
        s = specs[j]
        x, p = inputs[j]
        oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad)
        return s.flops(cfg["n"])

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    flops = sum(step(i) for i in range(args.steps))
    dt = time.perf_counter() - t
    v = flops / dt / 1e12
    return {"impl": "reference", "metric": "fused conv+BN+SiLU TFLOP/s & us/frame over the layer list; % of roofline",
            "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "layers": len(specs), "batch": cfg["n"],
                       "step": "one layer of the list per step, round robin"},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "one full-size layer of the list per step, round robin"},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="layer_list_fp32_n1", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    from conv_bn_silu_gb300 import build
    build.build()
    out = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
