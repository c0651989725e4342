"""One decode step per batch bucket, captured once as a CUDA graph and replayed.

A serving loop decodes a batch whose size and lengths change every step. The
kernels read the current lengths from device memory (decode_attn_splitk_dev),
so a step launched once for the longest contexts it will see stays valid while
the contexts grow; what a graph cannot follow is the batch size, because the
plan's work list is fixed at capture. So one graph is captured per bucket of
batch sizes (1, 2, 4, ... up to max_batch by default) and a step replays the
smallest bucket that holds the batch, with the rows past the batch given the
shortest valid length ("The Kernel Level: Attention and MoE", the CUDA-graph
section: static shapes, lengths in device memory, batch buckets).
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import api as A


def default_buckets(max_batch: int) -> List[int]:
    out, b = [], 1
    while b < max_batch:
        out.append(b)
        b *= 2
    out.append(max_batch)
    return out


class BucketedDecode:
    """Decode steps over a persistent cache, replayed from per-bucket CUDA graphs.

    q: [max_batch, Hq, Dk] (or [max_batch, q_len, Hq, Dk]) device buffer the caller
    fills with the step's queries; k_cache / v_cache: [max_batch, capacity, Hkv, D]
    (pass the same tensor twice and v_dim for MLA). Each bucket is planned for
    every sequence at `capacity` positions, so any lengths up to it are valid.
    Calling the object with the current lengths replays one graph and returns the
    first `batch` rows of the output buffer.
    """

    def __init__(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 scale: float, *, v_dim: Optional[int] = None,
                 out_dtype: torch.dtype = torch.float32,
                 buckets: Optional[Sequence[int]] = None):
        self.q, self.k, self.v = q, k_cache, v_cache
        self.max_batch = q.shape[0]
        self.q_len = q.shape[1] if q.dim() == 4 else 1
        self.capacity = k_cache.shape[1]
        self.buckets = sorted(set(buckets or default_buckets(self.max_batch)))
        if self.buckets[-1] > self.max_batch or self.buckets[0] < 1:
            raise ValueError("buckets must lie in [1, max_batch]")
        v_dim = v_cache.shape[3] if v_dim is None else int(v_dim)
        self.out = torch.empty(tuple(q.shape[:-1]) + (v_dim,), dtype=out_dtype, device=q.device)
        self.lens = torch.full((self.max_batch,), self.q_len, dtype=torch.int32, device=q.device)
        self.stream = torch.cuda.Stream(q.device)
        self.graphs, self._keep = {}, []
        self.stream.wait_stream(torch.cuda.current_stream(q.device))
        for b in self.buckets:
            a = A.make_args(q[:b], k_cache[:b], v_cache[:b], scale, v_dim=v_dim,
                            out_dtype=out_dtype)
            p = A.decode_attn_plan(a, [self.capacity] * b)
            ws = A.new_workspace(p, device=q.device)
            d = A.make_dev(seq_lens=self.lens[:b])
            out = self.out[:b]

            def step(a=a, p=p, ws=ws, d=d, out=out, b=b):
                # split, then the combine launch (the library's default)
                A.decode_attn_splitk_dev(a, p, d, q[:b], k_cache[:b], v_cache[:b], out, ws,
                                         self.stream)

            with torch.cuda.stream(self.stream):
                step()                                   # warm-up outside the capture
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    step()
            self.graphs[b] = g
            self._keep.append((a, p, ws, d))             # everything the graph points at
        torch.cuda.synchronize()

    def bucket_for(self, batch: int) -> int:
        for b in self.buckets:
            if b >= batch:
                return b
        raise ValueError(f"batch {batch} exceeds the largest bucket {self.buckets[-1]}")

    def __call__(self, seq_lens: Sequence[int] | torch.Tensor) -> torch.Tensor:
        """One step for the first len(seq_lens) sequences; returns out[:batch]
        (on this object's stream, which the caller's current stream waits for)."""
        batch = len(seq_lens)
        if batch < 1:
            raise ValueError("an empty batch")
        b = self.bucket_for(batch)
        cur = torch.cuda.current_stream(self.q.device)
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            lens = torch.as_tensor(seq_lens, dtype=torch.int32).to(self.q.device, non_blocking=True)
            self.lens[:batch].copy_(lens)
            if b > batch:
                self.lens[batch:b].fill_(self.q_len)     # padding rows: shortest valid length
            self.graphs[b].replay()
        cur.wait_stream(self.stream)
        return self.out[:batch]
