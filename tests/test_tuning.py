"""The measured plan table: lookup rules, and every entry plans on the host."""
import json

import pytest

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import tuning
from conv_bn_silu_gb300.layer import make_desc


def test_key_and_copy_rules(cuda_lib):
    d = make_desc(16, 64, 80, 80, 64, 3, 1, prec=B.CBS_BF16)
    key = tuning.shape_key(d)
    table = {key: {"force": {"force_block_m": 256, "force_k_group": 1, "force_block_n": 64}}}
    t = tuning.tuned_desc(d, table)
    assert (t.force_block_m, t.force_k_group, t.force_block_n) == (256, 1, 64)
    assert d.force_block_m == 0                      # the caller's descriptor is not modified
    # a descriptor that forces anything is left as it is
    f = make_desc(16, 64, 80, 80, 64, 3, 1, prec=B.CBS_BF16, force_block_n=32)
    assert tuning.tuned_desc(f, table) is f
    # other shapes (batch, layout, precision) do not match
    for other in (make_desc(1, 64, 80, 80, 64, 3, 1, prec=B.CBS_BF16),
                  make_desc(16, 64, 80, 80, 64, 3, 1, prec=B.CBS_TF32),
                  make_desc(16, 64, 80, 80, 64, 3, 1, prec=B.CBS_BF16, out_layout=B.CBS_NCHW)):
        assert tuning.shape_key(other) != key
        assert tuning.tuned_desc(other, table) is other
    with pytest.raises(ValueError):
        tuning.tuned_desc(d, {key: {"force": {"block_m": 1}}})


def test_every_table_entry_plans(cuda_lib):
    """The committed table's configurations are valid plans for their shapes."""
    table = tuning.load_table()
    for key, entry in table.items():
        prec, n, c_in, c_out, k, s, pad, h, w, il, ol = (int(v) for v in key.split(":"))
        d = make_desc(n, c_in, h, w, c_out, k, s, pad, prec=prec, in_layout=il, out_layout=ol)
        t = tuning.tuned_desc(d, table)
        p = B.cbs_plan(t)
        assert entry["us"] <= entry["auto_us"], key
        if "force_block_m" in entry["force"]:
            assert p.block_m == entry["force"]["force_block_m"], key


def test_table_file_is_well_formed():
    with open(tuning.TABLE_PATH) as f:
        meta = json.load(f)
    assert meta["created_by"] == "conv_bn_silu_gb300/autotune.py"
    assert isinstance(meta["plans"], dict)


def test_two_input_layers_are_keyed_apart():
    from conv_bn_silu_gb300 import _binding as B
    from conv_bn_silu_gb300.layer import make_desc
    from conv_bn_silu_gb300.tuning import shape_key, tuned_desc
    one = make_desc(16, 384, 40, 40, 128, 1, 1, prec=B.CBS_BF16)
    two = make_desc(16, 384, 40, 40, 128, 1, 1, prec=B.CBS_BF16, c_in_b=128)
    assert shape_key(one) != shape_key(two) and shape_key(two).endswith(":b128")
    table = {shape_key(one): {"force": {"force_block_n": 64}}}
    assert tuned_desc(one, table).force_block_n == 64
    assert tuned_desc(two, table).force_block_n == 0


def test_fp32_nhwc_candidates_force_the_variant(cuda_lib):
    """A forced tile field keeps an FP32 plan on the CUDA cores, so every
    autotune candidate for an FP32 NHWC shape names its variant too, and each
    one that plans lands on that variant (host-side, no GPU call)."""
    from conv_bn_silu_gb300 import autotune
    for prec, n, spec, lay in autotune.workload_shapes():
        if prec != "fp32" or lay != B.CBS_NHWC:
            continue
        base = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                         prec=B.CBS_FP32, in_layout=lay, out_layout=lay)
        for force in autotune.candidates(prec, spec, base):
            assert force.get("force_variant") == B.CBS_VARIANT_TC_TF32X3, force
            d = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                          prec=B.CBS_FP32, in_layout=lay, out_layout=lay, **force)
            try:
                pl = B.cbs_plan(d)
            except B.CbsError:
                continue
            assert pl.variant == B.CBS_VARIANT_TC_TF32X3
    # the table's FP32 NHWC entries force the variant as well
    for key, entry in tuning.load_table().items():
        fields = key.split(":")
        if fields[0] == str(B.CBS_FP32) and fields[9] == str(B.CBS_NHWC):
            assert entry["force"].get("force_variant") == B.CBS_VARIANT_TC_TF32X3, key


def test_fp32_nchw_flat_candidates_where_they_plan(cuda_lib):
    """The tuner offers flat NCHW boxes (force_window = 1, 3xTF32) exactly
    on the FP32 NCHW shapes the planner takes them for, and every such
    candidate that plans is a flat-box plan (host-side, no GPU call)."""
    from conv_bn_silu_gb300 import autotune
    seen_flat = seen_other = 0
    for prec, n, spec, lay in autotune.workload_shapes():
        if prec != "fp32" or lay != B.CBS_NCHW:
            continue
        base = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                         prec=B.CBS_FP32, in_layout=lay, out_layout=lay)
        cands = list(autotune.candidates(prec, spec, base))
        flat = [f for f in cands if f.get("force_window") == 1]
        eligible = (spec.c_in % 8 == 0 and spec.stride == 1 and spec.k == 2 * spec.pad + 1 and spec.pad <= 3
                    and spec.width % 4 == 0 and (n == 1 or (spec.oh * spec.ow) % 128 == 0))
        assert bool(flat) == eligible, (spec, n)
        seen_flat += bool(flat)
        seen_other += not flat
        for force in flat:
            assert force.get("force_variant") == B.CBS_VARIANT_TC_TF32X3, force
            d = make_desc(n, spec.c_in, spec.h, spec.width, spec.c_out, spec.k, spec.stride, spec.pad,
                          prec=B.CBS_FP32, in_layout=lay, out_layout=lay, **force)
            try:
                pl = B.cbs_plan(d)
            except B.CbsError as e:
                assert e.status == B.CBS_ERR_UNSUPPORTED, e   # K parts or N tile that do not fit
                continue
            assert pl.variant == B.CBS_VARIANT_TC_TF32X3 and pl.window == 1 and pl.k_group == 1
    assert seen_flat and seen_other   # both kinds occur among the list and chain shapes
