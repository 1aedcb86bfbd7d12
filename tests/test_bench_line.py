"""The bench's printed line stays small and carries the headline keys.

The full record (per-layer rows, the other workloads, the CPU baseline's
per-layer times) can run to tens of kilobytes; the printed line keeps only
what a reader of one line needs, so that a consumer keeping a short tail of
the output still sees all of it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def full_record():
    rows = [{"layer": i, "shape": "64->64 k3 s1 80", "us": 10.0, "mflop": 471.86} for i in range(40)]
    extra = {name: {"layers": rows, "ms_per_step": 0.3} for name in bench.EXTRA_DEFAULT}
    return {
        "metric": "fused conv+BN+SiLU TFLOP/s & us/frame over the layer list; % of roofline",
        "value": 14.1, "unit": "TFLOP/s", "n_gpus": 1, "steps": 20, "warmup": 5, "ms_per_step": 0.196,
        "us_per_frame": 196.0, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded N(0,1) inputs, He-init weights, random BN statistics)",
        "config": {"workload": "layer_list_fp32_n1", "layers": 12, "batch": 1, "layout": "NCHW",
                   "l2": "inputs larger than L2: 6 rotating copies of the step's 54.7 MB",
                   "timing": "x" * 300, "parallelism": "replicas x1", "launch": "programmatic dependent launch"},
        "roofline": {"bound": "alu", "kernel": "simt_conv_kernel (FP32 FMA), the 11 launches of one step",
                     "achieved": 11.1, "peak": 80.5, "unit": "TFLOP/s", "frac": 0.138,
                     "peak_source": "alu: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz (measured)",
                     "traffic": 28467456, "traffic_note": "y" * 100, "algorithmic_bytes": 43240000,
                     "sum_layer_roofline_us": 40.0, "frac_of_layer_roofline_sum": 0.2},
        "layers": rows, "per_step_us_with_launch_events": {"median": 1.0},
        "gpu_launches": 240,
        "e2e": {"value": 12.4, "unit": "TFLOP/s", "h2d_bytes_per_step": 27000000, "d2h_bytes_per_step": 27000000,
                "ms_per_step": 0.172, "steps": 20,
                "mode": ("4 steps in flight, each one copy in and one copy out "
                         "(inputs and outputs packed in one pinned buffer each way)"),
                "one_step_at_a_time": {"value": 8.0, "ms_per_step": 0.34}},
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "driver": "580", "samples": 30, "reasons": []},
        "peaks_source": "measured", "extra": extra,
        "cpu_baseline": {"value": 0.034, "unit": "TFLOP/s", "cores": 16, "kind": "oracle", "seconds": 10.2,
                         "machine": "aarch64", "sample": "120 full-size layers of the list at batch 1 (10 passes)",
                         "single_core": {"list_batch1_layer_ms": [1.0] * 12}},
    }


def test_compact_line_is_small_and_complete():
    out = full_record()
    line = json.dumps(bench.compact(out))
    assert len(line) < 2048, len(line)
    d = json.loads(line)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "cpu_baseline",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["config"]["workload"] == "layer_list_fp32_n1"
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in d["roofline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in d["e2e"], key
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in d["cpu_baseline"], key
    assert "layers" not in d and "extra" not in d


def test_traffic_figure_is_gated():
    """bench.py reports the recorded DRAM traffic only for the variant it was
    captured on and while the sources and plan-table entries hash to the
    recorded digest; a changed source or another dominant kernel gives null."""
    import bench
    t = bench.TRAFFIC["layer_list_fp32_n1"]
    assert bench.traffic_for("layer_list_fp32_n1", t["variant"]) == t["bytes"]
    assert bench.traffic_for("layer_list_fp32_n1", (t["variant"] + 1) % 6) is None
    assert bench.traffic_for("no_such_workload", t["variant"]) is None
    saved = dict(t)
    try:
        t["digest"] = "0" * 16
        assert bench.traffic_for("layer_list_fp32_n1", t["variant"]) is None
    finally:
        t.clear()
        t.update(saved)
    # the plan-table part of the digest covers only the workload's own entries
    d0 = bench.sources_digest(("../tuned_plans.json",))
    d1 = bench.sources_digest(("../tuned_plans.json",), table_prefix="2:", table_suffix=":1:1")
    assert d0 != d1
