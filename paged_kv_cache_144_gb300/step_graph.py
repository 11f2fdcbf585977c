"""One serving step recorded as a CUDA graph and replayed.

A decode step issues a few short launches (the cache write of the new
tokens, the decode, the copies of the step's inputs and result); issued one
by one from Python each costs host time (argument checks, marshalling, the
launch call), and for short steps that host time, not the GPU, sets the pace.
`StepGraph` records such a step once, with fixed buffers, through the same
library calls (the kernels, their programmatic dependent launches and the
copies become graph nodes), and `replay()` issues the whole step with one
graph launch.  The buffers must stay allocated and keep their addresses; new
inputs are written into them (host staging buffer, device tensors) before a
replay.
"""

from __future__ import annotations


class StepGraph:
    """Capture `fn` (a callable issuing the step's work on the current stream) as a CUDA graph.

    `warmup` eager calls run first on a side stream so that every launch plan and device symbol the calls
    look up is cached before capture (nothing may be looked up for the first time inside a capture).
    """

    def __init__(self, fn, *, warmup: int = 2):
        import torch
        self._torch = torch
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def replay(self):
        """Issue the recorded step on the current stream."""
        self.graph.replay()
