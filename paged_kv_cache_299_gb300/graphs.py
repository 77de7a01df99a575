"""CUDA-graph capture of a step of library calls ("vLLM", CUDA Graph: the decode forward is
captured once per batch size and replayed with a single launch instead of hundreds).

Every pa_* call of this library only enqueues kernels on the current stream and allocates
nothing (given a caller workspace), so a step built from them can be captured as is.  The
captured graph keeps the buffers' addresses: refresh their contents in place between
replays (new queries, new K/V, grown context lengths), never reallocate them.
"""
from __future__ import annotations

import torch


class StepGraph:
    """Capture `fn` (a closure over fixed device buffers) once; replay() re-runs it."""

    def __init__(self, fn, warmup: int = 1):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # first calls may set kernel attributes: not captured
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()

    def replay(self):
        self.graph.replay()


class GraphCache:
    """One StepGraph per key (typically the decode batch size), built on first use."""

    def __init__(self, make_step):
        self._make_step = make_step  # key -> closure enqueueing one step
        self._graphs = {}

    def run(self, key):
        g = self._graphs.get(key)
        if g is None:
            g = self._graphs[key] = StepGraph(self._make_step(key))
        g.replay()

    def __len__(self):
        return len(self._graphs)
