"""Measured per-shape plan table.

`cbs_plan` picks a tile configuration from a cost model, with no CUDA call
and no state.  On top of it, this module keeps a table of configurations
measured on GB300 for the layer shapes of the benchmark workloads: for a
(precision, batch, C_in, C_out, k, stride, pad, H, W, layouts) key it holds
the descriptor force fields of the fastest plan found by `autotune.py`.
`tuned_desc` fills those fields into a descriptor that forces nothing; a
descriptor that forces any field is left as it is, and shapes that are not in
the table keep the cost-model plan.
"""
from __future__ import annotations

import json
import os

from . import _binding as B

HERE = os.path.dirname(os.path.abspath(__file__))
TABLE_PATH = os.path.join(HERE, "tuned_plans.json")

# Descriptor fields a table entry may set.
FORCE_FIELDS = ("force_variant", "force_split_k", "force_block_n", "force_block_m", "force_k_group",
                "force_b_resident", "force_window", "force_issuer_split")
_DEFAULTS = {"force_variant": -1}

_table = None


def shape_key(d: B.cbs_layer_desc) -> str:
    key = ":".join(str(int(v)) for v in (d.prec, d.n, d.c_in, d.c_out, d.k, d.stride, d.pad, d.h, d.w,
                                         d.in_layout, d.out_layout))
    # A two-input layer plans its channel blocks around the junction of its
    # inputs: it is a shape of its own.
    return key + (f":b{int(d.c_in_b)}" if d.c_in_b else "")


def load_table(path: str = TABLE_PATH) -> dict:
    global _table
    if _table is None or path != TABLE_PATH:
        table = {}
        if os.path.exists(path):
            with open(path) as f:
                table = json.load(f).get("plans", {})
        if path != TABLE_PATH:
            return table
        _table = table
    return _table


def forces_nothing(d: B.cbs_layer_desc) -> bool:
    return all(int(getattr(d, f)) == _DEFAULTS.get(f, 0) for f in FORCE_FIELDS)


def tuned_desc(d: B.cbs_layer_desc, table: dict | None = None) -> B.cbs_layer_desc:
    """A copy of `d` with the measured configuration's force fields, if the
    table has its shape and `d` forces nothing; else `d` unchanged."""
    table = load_table() if table is None else table
    entry = table.get(shape_key(d))
    if entry is None or not forces_nothing(d):
        return d
    out = B.cbs_layer_desc.from_buffer_copy(d)
    for f, v in entry["force"].items():
        if f not in FORCE_FIELDS:
            raise ValueError(f"tuned plan table: unknown field {f}")
        setattr(out, f, int(v))
    return out
