"""Benchmark of the fused Conv2d + folded BN + SiLU layer on GB300.

Default workload: the twelve-layer YOLO26n-scale list at batch 1 in FP32,
NCHW in and out (the planner's choice per layer: the 3xTF32 tensor-core
kernel reading NCHW, the CUDA-core implicit GEMM, the direct stem kernel).  One step = the twelve fused layers,
each on its own seeded synthetic input, all resident in HBM.  The K timed
steps run as one captured CUDA graph (no host launch overhead inside the
timed region) with timing events between every kernel, so each launch's
device duration is measured in the same run.  Inputs and outputs rotate over
five copies (5 x 55 MB > the 126 MB L2), so no step finds its inputs in L2
from the step before.

Prints ONE compact JSON line (rank 0): the headline value, the roofline of
the dominant kernel, the end-to-end figure, the CPU baseline and the clocks.
`--detail PATH` writes the full record (per-layer rows; with `--extra`, the
other workloads too).  `--impl reference` times the CPU oracle on the host
cores on the same workload and metric instead.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from conv_bn_silu_gb300 import workloads as wl  # noqa: E402

# FP32 CUDA-core peak: SMs x 128 FP32 lanes x 2 FLOP per FMA x the maximum SM
# clock (GB300: 152 SMs, 2.07 GHz; both are read from the device when there is one).
DEFAULT_SMS, FP32_LANES, DEFAULT_SM_MAX_GHZ = 152, 128, 2.070
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
        driver = None
        try:
            driver = subprocess.run(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=driver_version",
                                     "--format=csv,noheader"], capture_output=True, text=True,
                                    timeout=10).stdout.strip() or None
        except (OSError, subprocess.SubprocessError):
            pass
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None, "driver": driver,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------- workloads
WORKLOADS = {
    "layer_list_fp32_n1": dict(kind="list", layers=wl.LAYER_LIST, n=1, prec="fp32"),
    "single_layer_fp32_n1": dict(kind="list", layers=(wl.SINGLE_LAYER,), n=1, prec="fp32"),
    "layer_list_bf16_n16": dict(kind="list", layers=wl.LAYER_LIST, n=16, prec="bf16"),
    "layer_list_tf32_n16": dict(kind="list", layers=wl.LAYER_LIST, n=16, prec="tf32"),
    "layer_list_int8_n16": dict(kind="list", layers=wl.LAYER_LIST, n=16, prec="int8"),
    "chain_fp32_n1": dict(kind="chain", n=1, prec="fp32"),
    "chain_bf16_n16": dict(kind="chain", n=16, prec="bf16"),
    "chain_tf32_n16": dict(kind="chain", n=16, prec="tf32"),
    "chain_fp32_n1_nhwc": dict(kind="chain", n=1, prec="fp32", layout="nhwc"),
    # The whole synthetic frame: the chain with the SPPF block (two more fused
    # layers and the three chained 5x5 pools in one glue kernel).
    "frame_fp32_n1": dict(kind="chain", n=1, prec="fp32", sppf=True),
    # The 40-layer chain on INT8 layers; and with the first layer (the raw
    # frame's) and the last kept in BF16, with quantise/dequantise seams.
    "chain_int8_n16": dict(kind="chain", n=16, prec="int8"),
    "chain_int8_n16_keepfloat": dict(kind="chain", n=16, prec="int8", keep_float=(0, 39)),
    "frame_bf16_n16": dict(kind="chain", n=16, prec="bf16", sppf=True),
    # The list with the residual form of the epilogue, y = SiLU(BN(conv)) + r, on every
    # stride-1 layer whose input and output shapes match (a bottleneck's skip add).
    "layer_list_bf16_n16_residual": dict(kind="list", layers=wl.LAYER_LIST, n=16, prec="bf16", residual=True),
    # asymmetric activations: input codes with zero point -20, outputs with -100
    "layer_list_int8_n16_asym": dict(kind="list", layers=wl.LAYER_LIST, n=16, prec="int8", zero_points=(-20, -100)),
    # FP32 with NHWC activations: layers with enough pixel tiles run the
    # 3xTF32 tensor-core kernel (the FP32 bar), the stem its direct kernel.
    "layer_list_fp32_n16_nhwc": dict(kind="list", layers=wl.LAYER_LIST, n=16, prec="fp32", layout="nhwc"),
    "layer_list_fp32_n1_nhwc": dict(kind="list", layers=wl.LAYER_LIST, n=1, prec="fp32", layout="nhwc"),
}
EXTRA_DEFAULT = ("layer_list_bf16_n16", "layer_list_tf32_n16", "layer_list_int8_n16", "chain_fp32_n1",
                 "chain_bf16_n16", "chain_tf32_n16", "layer_list_bf16_n16_residual", "layer_list_int8_n16_asym",
                 "layer_list_fp32_n16_nhwc", "layer_list_fp32_n1_nhwc", "chain_fp32_n1_nhwc", "frame_fp32_n1",
                 "frame_bf16_n16", "chain_int8_n16", "chain_int8_n16_keepfloat")


# DRAM traffic of the dominant kernel over one step of a workload, from one
# ncu capture of the default bench command's first warm-up step
# (dram__bytes_read.sum + dram__bytes_write.sum summed over that kernel's
# launches; the summary and command are in profiles/).  A figure is reported
# only while the kernel's sources and the measured plan table (which picks
# its tiles) are the ones the counters were taken from.
TRAFFIC = {
    # The 3xTF32 layers of the batch-1 FP32 list read their NCHW input in the
    # kernel (its converter warps gather it).
    "layer_list_fp32_n1": {"variant": 5, "kernel": "tc_conv_staged_kernel<TF32X3, NCHW gather>",
                           "launches": 9, "bytes": 24033536,
                           "sources": ("k_tc.cu", "cbs_api.cu", "cbs_internal.cuh", "../tuned_plans.json"),
                           "digest": "a9f4f1aa128cb01e",
                           "profile": "profiles/launches_layer_list_fp32_n1.md"},
}
# Variant of the dominant kernel per precision (the direct small-channel
# kernel runs the stem and is reported per layer, not here).
DOMINANT_VARIANT = {"fp32": 0, "tf32": 1, "bf16": 2, "int8": 3}
VARIANT_NAMES = {0: "simt_fp32", 1: "tc_tf32", 2: "tc_bf16", 3: "tc_int8", 4: "stem", 5: "tc_tf32x3"}
KERNEL_NAMES = {0: "simt_conv_kernel (FP32 FMA)", 1: "tc_conv_kernel<TF32>", 2: "tc_conv_kernel<BF16>",
                3: "tc_conv_staged_kernel<INT8>", 5: "tc_conv_staged_kernel<TF32X3> (FP32 as 3 TF32 products)"}
X3_VARIANT = 5


def sources_digest(files, table_prefix="0:", table_suffix=":0:0") -> str:
    """Hash of the kernel sources and, for the measured plan table, of the
    entries of the workload's shapes (by default FP32 with NCHW layouts: the
    key starts with the precision and ends with the two layouts); the other
    entries do not change these launches."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        path = os.path.join(ROOT, "conv_bn_silu_gb300", "csrc", f)
        if f.endswith("tuned_plans.json"):
            with open(path) as fh:
                plans = json.load(fh).get("plans", {})
            mine = {k: v for k, v in plans.items() if k.startswith(table_prefix) and k.endswith(table_suffix)}
            h.update(json.dumps(mine, sort_keys=True).encode())
            continue
        with open(path, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(workload: str, variant: int):
    t = TRAFFIC.get(workload)
    if t is None or t["variant"] != variant or sources_digest(t["sources"]) != t["digest"]:
        return None
    return t["bytes"]


def act_bytes(prec: str) -> int:
    return {"fp32": 4, "tf32": 4, "bf16": 2, "int8": 1}[prec]


def device_sms() -> int:
    try:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count)
    except Exception:
        pass
    return DEFAULT_SMS


def fp32_alu_peak(peaks):
    """(TFLOP/s, label): SMs x 128 lanes x 2 x the maximum SM clock."""
    sms = device_sms()
    ghz = float(peaks.get("sm_max_mhz", DEFAULT_SM_MAX_GHZ * 1e3)) / 1e3
    return sms * FP32_LANES * 2 * ghz / 1e3, f"alu: {sms} SMs x {FP32_LANES} FP32 lanes x 2 x {ghz:.3g} GHz"


def peak_for(prec: str, peaks):
    """(bound-kind peak in TFLOP/s, label) of the arithmetic a variant runs on."""
    bf16 = float(peaks["bf16_tflops"])
    if prec == "fp32":
        return fp32_alu_peak(peaks)
    if prec == "tf32":
        return bf16 * 1.1 / 2.25, "tensor: measured bf16 burst x nominal tf32/bf16 (1.1/2.25)"
    return bf16, "tensor: measured bf16 burst" + (" (int8 codes on bf16 MMA)" if prec == "int8" else "")


def int8_scales():
    path = os.path.join(ROOT, "tests", "golden", "int8_scales.json")
    return json.load(open(path))["layer_list"]


def int8_chain_scales():
    path = os.path.join(ROOT, "tests", "golden", "int8_chain_scales.json")
    return json.load(open(path))["chain"]


class ListWorkload:
    """Independent layers, each on its own resident input; inputs and outputs
    rotate over R copies so one rotation exceeds twice the L2 size."""

    def __init__(self, cfg, device):
        import torch
        from conv_bn_silu_gb300 import _binding as B
        from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc
        self.cfg, self.n, self.prec = cfg, cfg["n"], cfg["prec"]
        cp = {"fp32": B.CBS_FP32, "tf32": B.CBS_TF32, "bf16": B.CBS_BF16, "int8": B.CBS_INT8}[self.prec]
        self.specs = list(cfg["layers"])
        self.layers, host_x = [], []
        s_x = float(wl.S_X_INT8) if self.prec == "int8" else 0.0
        self.s_y = int8_scales() if self.prec == "int8" else [None] * len(self.specs)
        self.res = [bool(cfg.get("residual")) and s.c_in == s.c_out and s.stride == 1 for s in self.specs]
        z_x, z_y = cfg.get("zero_points", (0, 0))
        # FP32 reads NCHW as given unless the workload asks for NHWC; the
        # other precisions read the packed NHWC form.
        self.nhwc = self.prec != "fp32" or cfg.get("layout") == "nhwc"
        lay = B.CBS_NHWC if self.nhwc else B.CBS_NCHW
        for i, spec in enumerate(self.specs):
            x, p = wl.layer_inputs(spec, self.n, seed=0, layer_index=i)
            desc = make_desc(self.n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                             prec=cp, in_layout=lay, residual=int(self.res[i]), zero_point_x=z_x, zero_point_y=z_y)
            self.layers.append(FusedConvBnSilu(desc, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s_x=s_x,
                                               device=device))
            host_x.append(x)
        self.host_x = host_x
        ab = act_bytes(self.prec)
        # a residual layer also reads r (the output's size)
        self.extra_bytes = [self.n * s.c_out * s.oh * s.ow * ab if r else 0 for s, r in zip(self.specs, self.res)]
        self.step_bytes = sum(s.alg_bytes(self.n, ab) for s in self.specs) + sum(self.extra_bytes)
        self.R = max(2, int(np.ceil(2 * L2_BYTES / self.step_bytes)) + 1)
        packed = []
        for layer, x in zip(self.layers, host_x):
            xd = torch.from_numpy(x).to(device)
            packed.append(layer.pack_input(xd) if self.nhwc else xd)
        torch.cuda.synchronize()
        self.xs = [[t.clone() for t in packed] for _ in range(self.R)]
        self.ys = [[layer.empty_y() for layer in self.layers] for _ in range(self.R)]
        self.rs = [[layer.empty_y().normal_() if r else None for layer, r in zip(self.layers, self.res)]
                   for _ in range(self.R)]
        self.launches_per_step = len(self.layers)

    def step(self, r, stream_id, events=None, stream=None):
        for j, layer in enumerate(self.layers):
            if events is not None:
                events[j].record(stream)
            layer(self.xs[r % self.R][j], self.ys[r % self.R][j], s_y=self.s_y[j], stream=stream_id,
                  residual=self.rs[r % self.R][j])
        if events is not None:
            events[len(self.layers)].record(stream)

    def rows(self):
        return [(s, layer) for s, layer in zip(self.specs, self.layers)]


class ChainWorkload:
    """The 40-layer whole-frame chain, or the whole frame with the SPPF block;
    one step = one frame batch (frame packing, the fused layers, the upsample
    kernel and, in the frame, the SPPF pool kernel; two-input layers read
    their concatenated inputs straight from their buffers)."""

    def __init__(self, cfg, device):
        import torch
        from conv_bn_silu_gb300 import _binding as B
        from conv_bn_silu_gb300.chain import Chain
        self.cfg, self.n, self.prec = cfg, cfg["n"], cfg["prec"]
        lay = B.CBS_NHWC if cfg.get("layout") == "nhwc" else None
        kw = {}
        if self.prec == "int8":
            kw = dict(out_scales=int8_chain_scales(), keep_float=cfg.get("keep_float", ()))
        self.chain = Chain(self.prec, self.n, device=device, layout=lay, sppf=bool(cfg.get("sppf")), **kw)
        self.nhwc = self.chain.layout == B.CBS_NHWC
        self.frame = torch.from_numpy(wl.frame(self.n)).to(device)
        self.specs = [cl.spec for cl in self.chain.specs]
        self.layers = self.chain.layers
        self.step_bytes = self.chain.alg_bytes()
        self.R = 1
        self.launches_per_step = self.chain.launches_per_frame()

    def step(self, r, stream_id, events=None, stream=None):
        from conv_bn_silu_gb300 import _binding as B
        c = self.chain
        c.pack_frame(self.frame, stream_id)
        for i in range(len(c.layers)):
            c.glue_before(i, stream_id)
            if events is not None:
                events[i].record(stream)
            c.call(i, stream_id)
        if events is not None:
            events[len(c.layers)].record(stream)

    def rows(self):
        return [(s, layer) for s, layer in zip(self.specs, self.layers)]


def make_workload(name, device):
    cfg = WORKLOADS[name]
    return (ChainWorkload if cfg["kind"] == "chain" else ListWorkload)(cfg, device)


def measure(name, steps, warmup, device, peaks, sample_clocks=False):
    """Capture `steps` steps in one CUDA graph of plain launches (with the
    library's default programmatic dependent launch, consecutive kernels
    overlap their set-up), replay it once untimed, then once timed for the
    step time.  The same steps captured a second time with an external event
    between launches give each launch's duration (an event node between two
    kernels also orders them fully, so that replay is not the timed one)."""
    import torch
    w = make_workload(name, device)
    stream = torch.cuda.Stream(device)
    sid = stream.cuda_stream
    with torch.cuda.stream(stream):
        for i in range(warmup):
            w.step(i, sid)
    torch.cuda.synchronize()
    nl = len(w.layers)
    try:
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(nl + 1)] for _ in range(steps)]
    except TypeError:  # torch without external events: per-launch times unavailable
        evs = None
    def capture(events):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(steps):
                    w.step(i, sid, events[i] if events is not None else None, stream)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        return g

    graph = capture(None)
    graph_ev = capture(evs) if evs is not None else None
    sampler = ClockSampler(device.index) if sample_clocks else None
    if sampler:
        time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        graph.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    per_layer_us = None
    if evs is not None:
        with torch.cuda.stream(stream):
            graph_ev.replay()
        torch.cuda.synchronize()
        per_layer_us = np.zeros(nl)
        step_us = np.zeros(steps)
        for i in range(steps):
            for j in range(nl):
                per_layer_us[j] += evs[i][j].elapsed_time(evs[i][j + 1]) * 1e3
            step_us[i] = evs[i][0].elapsed_time(evs[i][nl]) * 1e3
        per_layer_us /= steps
    clocks = None
    if sampler:
        tend = time.time() + 1.0
        while time.time() < tend:
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize()
        clocks = sampler.stop()

    n, prec = w.n, w.prec
    ab = act_bytes(prec)
    peak, peak_label = peak_for(prec, peaks)
    hbm = float(peaks["hbm_gbs"])
    rows = []
    extra = getattr(w, "extra_bytes", None) or [0] * len(w.layers)
    for j, (sp, layer) in enumerate(w.rows()):
        f, by = sp.flops(n), sp.alg_bytes(n, ab) + extra[j]
        t_c, t_m = f / (peak * 1e12), by / (hbm * 1e9)
        bound = "compute" if t_c >= t_m else "hbm"
        if layer.plan.variant == X3_VARIANT:   # three TF32 products per multiply-add
            t_c = f / (peak_for("tf32", peaks)[0] / 3 * 1e12)
            bound = "compute" if t_c >= t_m else "hbm"
        row = {"layer": j + 1, "shape": f"{sp.c_in}->{sp.c_out} k{sp.k} s{sp.stride} {sp.h}" + (" +r" if extra[j] else ""),
               "variant": VARIANT_NAMES.get(layer.plan.variant, str(layer.plan.variant)),
               "tile": f"{layer.plan.block_m}x{layer.plan.block_n}", "split_k": layer.plan.split_k,
               "mflop": round(f / 1e6, 2), "alg_mb": round(by / 1e6, 3), "bound": bound,
               "roofline_us": round(max(t_c, t_m) * 1e6, 3), "compute_us": round(t_c * 1e6, 3)}
        if per_layer_us is not None:
            u = float(per_layer_us[j])
            row.update(us=round(u, 3), tflops=round(f / (u * 1e-6) / 1e12, 3),
                       frac_of_roofline=round(max(t_c, t_m) * 1e6 / u, 4),
                       frac_of_compute_peak=round(t_c * 1e6 / u, 4), frac_of_hbm=round(t_m * 1e6 / u, 4))
        rows.append(row)
    flops_step = sum(sp.flops(n) for sp in w.specs)
    ms_step = total_ms / steps
    kern_us = float(per_layer_us.sum()) if per_layer_us is not None else ms_step * 1e3
    out = {"workload": name, "prec": prec, "batch": n, "steps": steps, "ms_per_step": round(ms_step, 5),
           "tflops": round(flops_step / (ms_step * 1e-3) / 1e12, 4),
           "sum_layer_us": round(kern_us, 3),
           "sum_layer_roofline_us": round(sum(r["roofline_us"] for r in rows), 3),
           "frac_of_layer_roofline_sum": round(sum(r["roofline_us"] for r in rows) / kern_us, 4),
           "peak_tflops": round(peak, 2), "peak": peak_label, "hbm_gbs": hbm,
           "l2": (f"inputs larger than L2: {w.R} rotating copies of the step's {w.step_bytes / 1e6:.1f} MB"
                  if w.R > 1 else f"chain activations, {w.step_bytes / 1e6:.1f} MB algorithmic per frame batch"),
           "launches_per_step": w.launches_per_step, "layers": rows}
    if per_layer_us is not None:
        # Spread over the K steps of the per-launch replay (its event nodes
        # add ~5 us per launch, so these sit above ms_per_step).
        out["per_step_us_with_launch_events"] = {
            "median": round(float(np.median(step_us)), 2), "min": round(float(step_us.min()), 2),
            "p90": round(float(np.percentile(step_us, 90)), 2)}
    if per_layer_us is not None and name.startswith("layer_list") and n == 16:
        k3 = [r for r in rows if " k3 " in r["shape"] and r["bound"] == "compute"]
        mem = [r for r in rows if r not in k3]
        if k3:
            # each layer against the compute peak of the arithmetic its variant runs
            # (FP32 ALU, TF32, BF16, or TF32/3 for the 3xTF32 kernel)
            out["k3_compute_bound_frac_of_own_compute_peak"] = round(
                sum(r["compute_us"] for r in k3) / sum(r["us"] for r in k3), 4)
        if mem:
            out["hbm_bound_frac_of_hbm"] = round(
                sum(r["alg_mb"] for r in mem) * 1e6 / (sum(r["us"] for r in mem) * 1e-6) / (hbm * 1e9), 4)
    return out, w, clocks


def max_over_ranks(ms_step: float, device) -> float:
    """The job's step time: the slowest replica's (all_reduce MAX over the
    process group; NCCL on the GPUs, gloo in the CPU tests)."""
    import torch
    t = torch.tensor([ms_step], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_step: float, world: int, ms_step: float) -> float:
    """Whole-job throughput: every replica runs the same step (weak scaling),
    so the job does world x flops_step in the slowest replica's time."""
    return flops_step * world / (ms_step * 1e-3) / 1e12


def run_ours(args, rank: int, world: int):
    import torch
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(device)
    peaks, peak_src = load_peaks()
    from conv_bn_silu_gb300 import _binding as B
    B.cbs_set_launch_options(0 if args.no_pdl else B.CBS_LAUNCH_PDL)
    if world > 1:
        torch.distributed.barrier()
    head, w, clocks = measure(args.workload, args.steps, args.warmup, device, peaks, sample_clocks=True)
    if world > 1:
        torch.distributed.barrier()
    ms_step = head["ms_per_step"]
    if world > 1:
        ms_step = max_over_ranks(ms_step, device)
    n = w.n
    flops_step = sum(sp.flops(n) for sp in w.specs)
    value = job_tflops(flops_step, world, ms_step)
    rows = head["layers"]
    peak = head["peak_tflops"]
    # The dominant kernel: the variant (the stem's kernel aside) with the most
    # measured time in a step, and every layer the plans give to it.
    t_by_variant = {}
    for (sp, layer), r in zip(w.rows(), rows):
        if layer.plan.variant != B.CBS_VARIANT_STEM:
            t_by_variant[layer.plan.variant] = t_by_variant.get(layer.plan.variant, 0.0) + r["us"]
    dom_variant = max(t_by_variant, key=t_by_variant.get) if t_by_variant else DOMINANT_VARIANT[w.prec]
    kernel = KERNEL_NAMES[dom_variant]
    dom = [(sp, r) for (sp, layer), r in zip(w.rows(), rows) if layer.plan.variant == dom_variant]
    dom_flops = sum(sp.flops(n) for sp, _ in dom)
    dom_us = sum(r["us"] for _, r in dom)
    achieved = dom_flops / (dom_us * 1e-6) / 1e12
    traffic = traffic_for(args.workload, dom_variant)
    bound, peak_label = ("alu" if w.prec == "fp32" else "tensor"), head["peak"]
    if dom_variant == X3_VARIANT:   # FP32 as three TF32 products on the tensor cores
        peak = round(peak_for("tf32", peaks)[0] / 3, 2)
        bound, peak_label = "tensor", "tensor: measured bf16 burst x nominal tf32/bf16 (1.1/2.25) / 3 products"
    roofline = {"bound": bound,
                "kernel": f"{kernel}, the {len(dom)} launches of one step",
                "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_label + f" ({peak_src})",
                "traffic": traffic,
                "traffic_note": ((f"DRAM bytes in one step of {TRAFFIC[args.workload]['kernel']} (ncu, cold cache)")
                                 if traffic is not None else "no capture of the current kernel sources"),
                "algorithmic_bytes": sum(sp.alg_bytes(n, act_bytes(w.prec)) for sp, _ in dom),
                "sum_layer_roofline_us": head["sum_layer_roofline_us"],
                "frac_of_layer_roofline_sum": head["frac_of_layer_roofline_sum"]}
    e2e = run_e2e(w, device, args, flops_step, world)
    out = {
        "metric": "fused conv+BN+SiLU TFLOP/s & us/frame over the layer list; % of roofline",
        "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "us_per_frame": round(ms_step * 1e3 / n, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "tf32": "tf32", "bf16": "bf16", "int8": "int8"}[w.prec],
        "data": "synthetic (seeded N(0,1) inputs, He-init weights, random BN statistics)",
        "config": {"workload": args.workload, "layers": len(rows), "batch": n,
                   "layout": "NHWC" if getattr(w, "nhwc", w.prec != "fp32") else "NCHW", "l2": head["l2"],
                   "timing": ("K steps captured in one CUDA graph of programmatic dependent launches, CUDA events around "
                              "its replay on the launching stream; per-launch durations from a replay of the same K steps "
                              "captured with an event between launches"),
                   "parallelism": f"replicas x{world}",
                   "launch": "plain" if args.no_pdl else "programmatic dependent launch"},
        "roofline": roofline, "layers": rows,
        "per_step_us_with_launch_events": head.get("per_step_us_with_launch_events"),
        "gpu_launches": args.steps * w.launches_per_step,
        "e2e": e2e, "clocks": clocks, "peaks_source": peak_src,
    }
    if rank == 0 and args.extra:
        extra = {}
        for name in EXTRA_DEFAULT:
            if name == args.workload:
                continue
            try:
                summ, _, _ = measure(name, min(args.steps, 20), 3, device, peaks)
                extra[name] = summ
            except Exception as exc:  # report, do not hide, a failing extra workload
                extra[name] = {"error": f"{type(exc).__name__}: {exc}"}
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        out["extra"] = extra
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    return out


def compact(out: dict) -> dict:
    """The one JSON line the bench prints: the headline figures only (a few
    hundred bytes).  Per-layer rows, the other workloads' summaries and the
    CPU baseline's per-layer times go to the --detail file."""
    rf = out["roofline"]
    line = {k: out[k] for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                                "us_per_frame", "higher_is_better", "scaling", "vs_baseline", "dtype", "data")}
    cfg = out["config"]
    line["config"] = {k: cfg[k] for k in ("workload", "layers", "batch", "layout", "l2", "parallelism", "launch")}
    line["roofline"] = {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    line["roofline"].update(kernel=rf["kernel"], algorithmic_bytes=rf["algorithmic_bytes"],
                            peak_source=rf["peak_source"],
                            frac_of_layer_roofline_sum=rf["frac_of_layer_roofline_sum"])
    e = out["e2e"]
    line["e2e"] = {k: e[k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "ms_per_step",
                                     "mode") if k in e}
    cb = out.get("cpu_baseline")
    if cb is not None:
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "machine")}
    line["gpu_launches"] = out["gpu_launches"]
    ck = out.get("clocks") or {}
    line["clocks"] = {k: ck.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    return line


def run_e2e(w, device, args, flops_step, world):
    """Same metric through the public API with host buffers: each step copies
    its inputs from pinned host memory (FP32 activations for the FP32 list;
    the packed input format otherwise), runs the layers and reads every output
    back.  Each step is one CUDA graph (conv_bn_silu_gb300.host_io).  The
    reported value runs four steps in flight on four buffer sets (each with
    layers of its own split-K workspaces).  A set keeps the step's inputs,
    and its outputs, as views of one buffer each way, so a step is one copy
    in, the twelve layers back to back (their programmatic dependent
    launches intact) and one copy out; the copies overlap the neighbouring
    steps' kernels.  Measured on GB300 for the FP32 list:
      0.171-0.174 ms per step, about the device-resident step;
      0.209-0.211 ms with one copy per tensor;
      0.220-0.222 ms with two sets and each layer's copies overlapping the
        same step's other layers, whose per-layer events break the kernels'
        programmatic dependent launches.
    A list with fewer than three buffer sets runs two steps in flight with
    per-layer overlap.  The one-step-at-a-time figure, where the host waits
    for every step's result, is reported beside it.  The chain copies its
    frame in and its last output out, one step at a time."""
    import torch
    from conv_bn_silu_gb300.host_io import HostPipeline
    stream = torch.cuda.Stream(device)
    sid = stream.cuda_stream
    xs_d = w.xs[0] if hasattr(w, "xs") else [w.frame]
    ys_d = w.ys[0] if hasattr(w, "ys") else [w.chain.outs[-1]]
    xs_h = [x.cpu().pin_memory() for x in xs_d]
    ys_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in ys_d]
    steps = max(3, min(args.steps, 50))

    pipelined = None
    if hasattr(w, "xs"):
        from conv_bn_silu_gb300.host_io import DoubleBufferedRunner, pack_layout, packed_views

        def capture_set(r, xh, yh, per_layer=True, own_workspaces=False):
            # Steps in flight together run the same layers at once: each
            # buffer set then takes layers with workspaces of their own.
            layers = [layer.fork() for layer in w.layers] if own_workspaces else w.layers
            xd, yd = w.xs[r], w.ys[r]
            calls = [(lambda st, j=j: layers[j](xd[j], yd[j], s_y=w.s_y[j], stream=st, residual=w.rs[r][j]))
                     for j in range(len(layers))]
            return HostPipeline(len(layers), device, per_layer=per_layer).capture(calls, xh, xd, yd, yh)

        def host_set():
            return ([x.clone().pin_memory() for x in xs_h],
                    [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in ys_h])

        x_off, x_total = pack_layout(xs_d)
        y_off, y_total = pack_layout(ys_d)

        def capture_packed_set(r):
            # The step's inputs and outputs as views of one device buffer
            # each, filled from and read back to one pinned host buffer each.
            layers = [layer.fork() for layer in w.layers]
            xd = torch.empty(x_total, dtype=torch.uint8, device=device)
            yd = torch.empty(y_total, dtype=torch.uint8, device=device)
            xh = torch.empty(x_total, dtype=torch.uint8).pin_memory()
            yh = torch.empty(y_total, dtype=torch.uint8).pin_memory()
            for v, x in zip(packed_views(xh, xs_h, x_off), xs_h):
                v.copy_(x)
            xv, yv = packed_views(xd, xs_d, x_off), packed_views(yd, ys_d, y_off)

            def call(st):
                for j in range(len(layers)):
                    layers[j](xv[j], yv[j], s_y=w.s_y[j], stream=st, residual=w.rs[r][j])
            return HostPipeline(1, device, per_layer=False).capture([call], [xh], [xd], [yd], [yh])

        one = capture_set(0, xs_h, ys_h)
        packed_sets = 0
        if w.R >= 3:
            packed_sets = min(4, w.R)
            pipelined = DoubleBufferedRunner([capture_packed_set(r) for r in range(packed_sets)])
            pipe_mode = (f"{packed_sets} steps in flight, each one copy in and one copy out "
                         "(inputs and outputs packed in one pinned buffer each way)")
        elif w.R >= 2:
            pipelined = DoubleBufferedRunner([capture_set(r, *host_set(), own_workspaces=True) for r in range(2)])
            pipe_mode = "two steps in flight, double-buffered host I/O"
        torch.cuda.synchronize()   # the forked workspaces are initialised on the current stream
    else:
        def one():
            with torch.cuda.stream(stream):
                for j in range(len(xs_d)):
                    xs_d[j].copy_(xs_h[j], non_blocking=True)
                w.step(0, sid)
                for j in range(len(ys_d)):
                    ys_h[j].copy_(ys_d[j], non_blocking=True)
            stream.synchronize()

    for _ in range(3):
        one()
    t = time.perf_counter()
    for _ in range(steps):
        one()
    dt_sync = (time.perf_counter() - t) / steps
    h2d = sum(x.numel() * x.element_size() for x in xs_h)
    d2h = sum(y.numel() * y.element_size() for y in ys_h)
    if pipelined is not None and packed_sets:
        h2d, d2h = x_total, y_total   # the packed buffers, alignment gaps included
    out = {"h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps, "unit": "TFLOP/s"}
    if pipelined is not None:
        # Throughput with several steps in flight (a buffer set each): every
        # step still copies its inputs in and its outputs out inside the
        # timed region; the host waits once, at the end.
        pipelined.run(4)
        t = time.perf_counter()
        pipelined.run(steps)
        dt = (time.perf_counter() - t) / steps
        out.update(value=round(flops_step * world / dt / 1e12, 4), ms_per_step=round(dt * 1e3, 4),
                   mode=pipe_mode,
                   one_step_at_a_time={"value": round(flops_step * world / dt_sync / 1e12, 4),
                                       "ms_per_step": round(dt_sync * 1e3, 4)})
    else:
        out.update(value=round(flops_step * world / dt_sync / 1e12, 4), ms_per_step=round(dt_sync * 1e3, 4),
                   mode="one step at a time")
    return out


def cpu_baseline(w, budget_s: float = 10.0):
    """The CPU oracle as it stands, on the host cores, on a bounded sample of
    the same workload: passes over the list's layers (full size) until about
    `budget_s` seconds of CPU work are done."""
    import oracle
    specs = list(WORKLOADS["layer_list_fp32_n1"]["layers"]) if not hasattr(w, "host_x") else w.specs
    n = w.n if hasattr(w, "host_x") else 1
    inputs = [wl.layer_inputs(s, n, seed=0, layer_index=i) for i, s in enumerate(specs)]
    done_flops, layers_done, t0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        for spec, (x, p) in zip(specs, inputs):
            oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, spec.stride, spec.pad)
            done_flops += spec.flops(n)
            layers_done += 1
    dt = time.perf_counter() - t0
    cores = oracle.num_threads()
    out = {"value": round(done_flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
           "kind": "oracle", "seconds": round(dt, 2), "machine": platform.machine(),
           "sample": f"{layers_done} full-size layers of the list at batch {n} "
                     f"({layers_done / len(specs):.0f} passes), double arithmetic"}
    # The same oracle on one core: the single layer (config 1) and one pass
    # over the batch-1 list, per layer.
    oracle.set_threads(1)
    try:
        s1 = wl.SINGLE_LAYER
        x1, p1 = wl.layer_inputs(s1, 1)
        t = time.perf_counter()
        for _ in range(3):
            oracle.conv_bn_silu_f32(x1, p1.w, p1.gamma, p1.beta, p1.mean, p1.var, p1.eps, s1.stride, s1.pad)
        single_ms = (time.perf_counter() - t) / 3 * 1e3
        list_specs = list(WORKLOADS["layer_list_fp32_n1"]["layers"])
        per_layer = []
        for i, s in enumerate(list_specs):
            x, p = wl.layer_inputs(s, 1, seed=0, layer_index=i)
            t = time.perf_counter()
            oracle.conv_bn_silu_f32(x, p.w, p.gamma, p.beta, p.mean, p.var, p.eps, s.stride, s.pad)
            per_layer.append(round((time.perf_counter() - t) * 1e3, 2))
        out["single_core"] = {"single_layer_ms": round(single_ms, 2), "list_batch1_layer_ms": per_layer,
                              "list_batch1_tflops": round(sum(sp.flops(1) for sp in list_specs)
                                                          / (sum(per_layer) * 1e-3) / 1e12, 6)}
    finally:
        oracle.set_threads(cores)
    return out


def run_reference(args, rank: int, world: int):
    """The oracle on the host cores: each step is one layer of the list
    (round robin), full size."""
    if rank != 0:
        return None
    import oracle
    cfg = WORKLOADS[args.workload]
    specs = cfg["layers"] if cfg["kind"] == "list" else [cl.spec for cl in wl.chain_layers()]
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
    ap.add_argument("--extra", action="store_true",
                    help="also measure the other workloads (summaries go to the --detail file)")
    ap.add_argument("--no-extra", action="store_true", help="(default) measure the chosen workload only")
    ap.add_argument("--detail", default=None,
                    help="write the full record (per-layer rows, clocks, extras, CPU baseline detail) "
                         "as JSON to this path")
    ap.add_argument("--no-pdl", action="store_true",
                    help="plain launches instead of programmatic dependent launches (for comparison)")
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
        if args.detail:
            d = os.path.dirname(os.path.abspath(args.detail))
            os.makedirs(d, exist_ok=True)
            with open(args.detail, "w") as fh:
                json.dump(out, fh, indent=1)
        print(json.dumps(compact(out)), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
