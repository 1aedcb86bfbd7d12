"""Fused Conv2d + folded BatchNorm + SiLU for GB300 (sm_103a).

The computation lives in libcbs.so (C ABI in include/cbs.h, CUDA kernels in
csrc/).  This package is its thin Python binding: `_binding` exposes the C
calls under their own names, `layer` adds PyTorch device buffers and streams,
`workloads` holds the seeded synthetic inputs the tests and the benchmark use.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import CbsError, lib  # noqa: F401
