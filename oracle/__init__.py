"""CPU oracle for the fused Conv2d + BatchNorm + SiLU layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library under
``conv_bn_silu_gb300`` never does, and the two share no code.
"""
from .oracle import (  # noqa: F401
    out_dim,
    conv2d,
    batchnorm,
    silu,
    conv_bn_silu_f32,
    conv_bn_act_f32,
    maxpool2d_f32,
    spec_exp,
    spec_exp_max_rel_err,
    quantize_act,
    dequantize_i8,
    round_bf16,
    fold_quant_i8,
    requant,
    requant_array,
    conv_i8,
    num_threads,
    set_threads,
)
