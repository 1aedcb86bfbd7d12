"""Layers on host-resident tensors, with the copies overlapped with the kernels.

For a run of independent layers whose inputs and outputs live in pinned host
memory, `HostPipeline.run` enqueues
  - every host-to-device input copy, back to back, on a copy stream;
  - layer j on the compute stream, after an event that marks its own input
    as landed (not after all inputs);
  - layer j's device-to-host output copy on a second copy stream, as soon as
    an event marks the layer as finished;
so the host link carries inputs and outputs in both directions while the
kernels run, instead of copy-all / compute-all / copy-all.  With
`per_layer=False` a step is copy-all / compute-all / copy-all after all:
the kernels then follow one another with no event between them (the
library's programmatic dependent launches overlap their set-up), and the
copies overlap the neighbouring steps' kernels instead.
`DoubleBufferedRunner` runs such steps in turn over two or more buffer
sets, so one step's copies also overlap the neighbouring steps' kernels.
Steps in flight together need layers with workspaces of their own
(`FusedConvBnSilu.fork`).  `pack_layout` and `packed_views` place a step's
inputs (or outputs) in one buffer, so the step moves them with one copy
each way.  The copies are cudaMemcpyAsync calls (torch's copy_ on pinned
memory) and every layer is a library kernel: nothing is computed on the
host.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch


class HostPipeline:
    def __init__(self, n_layers: int, device="cuda", per_layer: bool = True):
        device = torch.device(device)
        self.per_layer = per_layer
        self.h2d = torch.cuda.Stream(device)
        self.compute = torch.cuda.Stream(device)
        self.d2h = torch.cuda.Stream(device)
        self.ev_in = [torch.cuda.Event() for _ in range(n_layers)]
        self.ev_out = [torch.cuda.Event() for _ in range(n_layers)]

    def _enqueue(self, calls, xs_h, xs_d, ys_d, ys_h, origin) -> None:
        n = len(calls)
        assert n <= len(self.ev_in) and len(xs_h) == len(xs_d) == n and len(ys_d) == len(ys_h) == n
        # Work already queued on `origin` may still use these buffers.
        self.h2d.wait_stream(origin)
        self.compute.wait_stream(origin)
        self.d2h.wait_stream(origin)
        with torch.cuda.stream(self.h2d):
            for j in range(n):
                xs_d[j].copy_(xs_h[j], non_blocking=True)
                self.ev_in[j].record(self.h2d)
        sid = self.compute.cuda_stream
        if not self.per_layer:
            self.compute.wait_event(self.ev_in[n - 1])   # the copies run in order: all inputs landed
            for j in range(n):
                calls[j](sid)
            self.ev_out[n - 1].record(self.compute)
            self.d2h.wait_event(self.ev_out[n - 1])
            with torch.cuda.stream(self.d2h):
                for j in range(n):
                    ys_h[j].copy_(ys_d[j], non_blocking=True)
            return
        for j in range(n):
            self.compute.wait_event(self.ev_in[j])
            calls[j](sid)
            self.ev_out[j].record(self.compute)
            self.d2h.wait_event(self.ev_out[j])
            with torch.cuda.stream(self.d2h):
                ys_h[j].copy_(ys_d[j], non_blocking=True)

    def run(self, calls: Sequence[Callable[[int], None]], xs_h, xs_d, ys_d, ys_h) -> None:
        """calls[j](stream) launches layer j on `stream` (a cudaStream_t as
        int), reading xs_d[j] and writing ys_d[j].  xs_h / ys_h: pinned host
        tensors of the same shapes.  Returns once every output is in ys_h."""
        self._enqueue(calls, xs_h, xs_d, ys_d, ys_h, torch.cuda.current_stream())
        self.d2h.synchronize()

    def capture(self, calls: Sequence[Callable[[int], None]], xs_h, xs_d, ys_d, ys_h) -> Callable[[], None]:
        """The same work recorded once as a CUDA graph (copies, kernels and
        the events between the three streams become graph nodes and edges),
        so a step costs one launch on the host.  Returns a function that
        replays it and returns once every output is in ys_h; the function
        holds every tensor the graph uses.  Steps that may run at the same
        time (DoubleBufferedRunner) need their own layer workspaces
        (FusedConvBnSilu.fork)."""
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(self.compute.device)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(graph, stream=cap):
            self._enqueue(calls, xs_h, xs_d, ys_d, ys_h, cap)   # fork from the capture stream
            cap.wait_stream(self.h2d)                          # join every stream back
            cap.wait_stream(self.compute)
            cap.wait_stream(self.d2h)

        def replay(wait: bool = True) -> None:
            with torch.cuda.stream(cap):
                graph.replay()
            if wait:
                cap.synchronize()
        replay.stream = cap
        # The graph's copy and kernel nodes hold raw addresses of these
        # tensors (and of whatever `calls` closes over): they live as long
        # as the replay does.
        replay.keep = (graph, calls, xs_h, xs_d, ys_d, ys_h)
        return replay


def pack_layout(like: Sequence[torch.Tensor], align: int = 256):
    """Byte offsets that place tensors shaped like `like` one after another
    in one buffer, each start a multiple of `align` bytes (the kernels' TMA
    loads need 16), and the buffer's total size."""
    offsets, off = [], 0
    for t in like:
        offsets.append(off)
        off += -(-t.numel() * t.element_size() // align) * align
    return offsets, off


def packed_views(buf: torch.Tensor, like: Sequence[torch.Tensor], offsets) -> list:
    """Views of the uint8 tensor `buf` at `offsets` with the shapes and
    dtypes of `like`.  A step whose inputs (or outputs) are such views of
    one buffer moves them with one copy each way, which the host link
    carries faster than one copy per tensor."""
    return [buf.narrow(0, o, t.numel() * t.element_size()).view(t.dtype).view(t.shape)
            for t, o in zip(like, offsets)]


class DoubleBufferedRunner:
    """Back-to-back steps with two (or more) sets of buffers: step i uses set
    i % len(replays), and
    each set's captured step (HostPipeline.capture) replays on its own stream,
    so step i + 1's input copies run while step i computes and its outputs
    are read back.  A set's next step starts only after its previous one has
    finished (same stream), so no buffer is overwritten while in use."""

    def __init__(self, replays):
        assert len(replays) >= 2
        self.replays = replays

    def run(self, steps: int) -> None:
        """Enqueue `steps` steps, then wait until every output is on the host."""
        for i in range(steps):
            self.replays[i % len(self.replays)](wait=False)
        for r in self.replays:
            r.stream.synchronize()
