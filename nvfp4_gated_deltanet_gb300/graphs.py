"""Per-bucket CUDA graphs of the decode step.

Rocket blog, "A reduction barrier makes Qwen GDN graph replay bit exact": one
immutable graph per decode bucket (c1, c2, c4, c8, c16), captured once and
replayed, with runtime dispatch removed from the replayed path. Here each
bucket's graph holds the launches of one gdn_decode_step on static buffers;
a step is: write x and slot ids into the static buffers, replay the bucket.
Rows whose slot id is -1 are padding (zero output, no state touched), so a
batch of n sequences runs in the smallest bucket >= n.
"""
from __future__ import annotations

import torch


class DecodeGraphs:
    def __init__(self, layer, conv_state, ssm_state, buckets=(1, 2, 4, 8, 16), max_batch=None, device="cuda"):
        self.layer = layer
        self.conv_state, self.ssm_state = conv_state, ssm_state
        self.buckets = sorted(buckets)
        mb = max_batch or self.buckets[-1]
        self.x = torch.zeros(mb, layer.H, dtype=torch.int16, device=device)
        self.slot_ids = torch.full((mb,), -1, dtype=torch.int32, device=device)
        self.out = torch.zeros(mb, layer.H, dtype=torch.int16, device=device)
        self.graphs = {}
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for B in self.buckets:          # warm-up launch outside capture (all rows padding)
                self._step(B)
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        for B in self.buckets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._step(B)
            self.graphs[B] = g
        torch.cuda.synchronize()

    def _step(self, B):
        self.layer.decode_step(self.x[:B], self.slot_ids[:B], self.conv_state, self.ssm_state, out=self.out[:B])

    def bucket_for(self, n: int) -> int:
        for B in self.buckets:
            if B >= n:
                return B
        raise ValueError(f"batch {n} exceeds the largest bucket {self.buckets[-1]}")

    def replay(self, B: int):
        self.graphs[B].replay()

    def step(self, x: torch.Tensor, slot_ids: torch.Tensor) -> torch.Tensor:
        """Run n = len(slot_ids) rows in the smallest bucket; returns out[:n]."""
        n = x.shape[0]
        B = self.bucket_for(n)
        self.x[:n].copy_(x)
        self.slot_ids[:n].copy_(slot_ids)
        if B > n:
            self.slot_ids[n:B].fill_(-1)
        self.replay(B)
        return self.out[:n]


class DecodeStackGraph:
    """One CUDA graph of a decode step through several layers (each with its
    own weights and states), for a fixed row count B: layer i reads x[i] and
    writes out[i]. A step is: write x (e.g. from pinned host memory), replay,
    read out -- one graph launch instead of three kernel launches per layer
    from the host, as in a served stack whose per-bucket graph holds every
    layer."""

    def __init__(self, layers, states, B: int, device="cuda"):
        self.layers, self.states, self.B = list(layers), list(states), B
        H = self.layers[0].H
        n = len(self.layers)
        self.x = torch.zeros(n, B, H, dtype=torch.int16, device=device)
        self.out = torch.zeros(n, B, H, dtype=torch.int16, device=device)
        self.slot_ids = torch.arange(B, dtype=torch.int32, device=device)
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):  # warm-up launch outside capture
            self._launch()
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._launch()
        torch.cuda.synchronize()

    def _launch(self):
        for i, (L, (c, m)) in enumerate(zip(self.layers, self.states)):
            L.decode_step(self.x[i], self.slot_ids, c, m, out=self.out[i])

    def replay(self):
        self.graph.replay()

    def step(self, x: torch.Tensor) -> torch.Tensor:
        """x [n_layers][B][H] (any device; copied without a host sync) -> out."""
        self.x.copy_(x, non_blocking=True)
        self.replay()
        return self.out
