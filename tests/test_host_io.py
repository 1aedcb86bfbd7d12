"""GPU check of the host-I/O pipeline: layers run on pinned host tensors
(copies overlapped with the kernels on separate streams) give exactly the
outputs of the same layers run on device-resident tensors, run after run."""
import pytest
import torch

from conv_bn_silu_gb300 import _binding as B
from conv_bn_silu_gb300 import workloads as wl
from conv_bn_silu_gb300.host_io import HostPipeline
from conv_bn_silu_gb300.layer import FusedConvBnSilu, make_desc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("per_layer", [True, False])
@pytest.mark.parametrize("prec", [B.CBS_FP32, B.CBS_BF16])
def test_pipeline_matches_device_runs(cuda_lib, prec, per_layer):
    specs = [wl.LayerSpec(16, 32, 3, 2, 64), wl.LayerSpec(32, 32, 1, 1, 40), wl.LayerSpec(64, 128, 3, 1, 20)]
    layers, xs_d = [], []
    for i, s in enumerate(specs):
        x, p = wl.layer_inputs(s, 2, layer_index=30 + i)
        layer = FusedConvBnSilu(make_desc(2, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad, prec=prec),
                                p.w, p.gamma, p.beta, p.mean, p.var, p.eps)
        xd = torch.from_numpy(x).cuda()
        xs_d.append(layer.pack_input(xd) if prec != B.CBS_FP32 else xd)
        layers.append(layer)
    want = [layer(x).cpu() for layer, x in zip(layers, xs_d)]
    xs_h = [x.cpu().pin_memory() for x in xs_d]
    ys_d = [layer.empty_y() for layer in layers]
    ys_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in ys_d]
    pipe = HostPipeline(len(layers), per_layer=per_layer)
    calls = [(lambda st, j=j: layers[j](xs_d[j], ys_d[j], stream=st)) for j in range(len(layers))]
    replay = pipe.capture(calls, xs_h, xs_d, ys_d, ys_h)
    for run in range(6):
        for y in ys_h:
            y.zero_()
        for x in xs_d:          # the pipeline must bring the inputs in itself
            x.zero_()
        torch.cuda.synchronize()
        if run % 2:
            replay()            # the CUDA-graph form
        else:
            pipe.run(calls, xs_h, xs_d, ys_d, ys_h)
        for j in range(len(layers)):
            assert torch.equal(ys_h[j], want[j]), (run, j)


@pytest.mark.parametrize("sets,per_layer", [(2, True), (3, False)])
def test_double_buffered_runner(cuda_lib, sets, per_layer):
    """Two or three buffer sets, as many steps in flight: every step's
    outputs reach the host and equal a device-resident run."""
    from conv_bn_silu_gb300.host_io import DoubleBufferedRunner
    s = wl.LayerSpec(32, 64, 3, 1, 40)
    x, p = wl.layer_inputs(s, 2, layer_index=40)
    layer = FusedConvBnSilu(make_desc(2, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad), p.w, p.gamma,
                            p.beta, p.mean, p.var, p.eps)
    want = layer(torch.from_numpy(x).cuda()).cpu()
    replays, hosts = [], []
    for r in range(sets):
        xd, yd = [torch.from_numpy(x).cuda()], [layer.empty_y()]
        xh, yh = [torch.from_numpy(x).pin_memory()], [torch.empty(yd[0].shape).pin_memory()]
        mine = layer.fork()   # steps in flight together: a split-K workspace each
        calls = [lambda st, xd=xd, yd=yd, mine=mine: mine(xd[0], yd[0], stream=st)]
        replays.append(HostPipeline(1, per_layer=per_layer).capture(calls, xh, xd, yd, yh))
        hosts.append(yh[0])
    torch.cuda.synchronize()   # the forked workspaces are initialised on the current stream
    runner = DoubleBufferedRunner(replays)
    for steps in (1, 2, 7):
        for h in hosts:
            h.zero_()
        runner.run(steps)
        for r in range(min(steps, sets)):
            assert torch.equal(hosts[r], want), (steps, r)


def test_packed_sets_match_device_runs(cuda_lib):
    """Three buffer sets in flight, each step's inputs and outputs packed in
    one buffer per direction (one copy each way), the layers forked per set:
    every set's outputs equal device-resident runs."""
    from conv_bn_silu_gb300.host_io import DoubleBufferedRunner, pack_layout, packed_views
    specs = [wl.LayerSpec(16, 32, 3, 2, 64), wl.LayerSpec(32, 48, 3, 1, 40), wl.LayerSpec(64, 64, 1, 1, 20)]
    layers, xs = [], []
    for i, s in enumerate(specs):
        x, p = wl.layer_inputs(s, 1, layer_index=50 + i)
        layers.append(FusedConvBnSilu(make_desc(1, s.c_in, s.h, s.width, s.c_out, s.k, s.stride, s.pad),
                                      p.w, p.gamma, p.beta, p.mean, p.var, p.eps))
        xs.append(torch.from_numpy(x))
    want = [layer(x.cuda()).cpu() for layer, x in zip(layers, xs)]
    ys_like = [layer.empty_y() for layer in layers]
    x_off, x_total = pack_layout(xs)
    y_off, y_total = pack_layout(ys_like)
    replays, outs = [], []
    for r in range(3):
        mine = [layer.fork() for layer in layers]
        xd = torch.zeros(x_total, dtype=torch.uint8, device="cuda")
        yd = torch.zeros(y_total, dtype=torch.uint8, device="cuda")
        xh = torch.empty(x_total, dtype=torch.uint8).pin_memory()
        yh = torch.empty(y_total, dtype=torch.uint8).pin_memory()
        for v, x in zip(packed_views(xh, xs, x_off), xs):
            v.copy_(x)
        xv, yv = packed_views(xd, xs, x_off), packed_views(yd, ys_like, y_off)

        def call(st, mine=mine, xv=xv, yv=yv):
            for j in range(len(mine)):
                mine[j](xv[j], yv[j], stream=st)
        replays.append(HostPipeline(1, per_layer=False).capture([call], [xh], [xd], [yd], [yh]))
        outs.append(packed_views(yh, ys_like, y_off))
    torch.cuda.synchronize()
    runner = DoubleBufferedRunner(replays)
    for steps in (3, 8):
        for o in outs:
            for t in o:
                t.zero_()
        runner.run(steps)
        for r in range(3):
            for j in range(len(layers)):
                assert torch.equal(outs[r][j], want[j]), (steps, r, j)
    assert B.cbs_read_device_status(True, torch.cuda.current_stream().cuda_stream) == B.CBS_OK
