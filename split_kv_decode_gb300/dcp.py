"""Context-parallel decode (DCP) across ranks.

Each rank holds a contiguous slice of every sequence's KV cache. It runs the
split kernel on its slice, the ranks all-gather their partials, and every rank
merges them with the same exp(m_i - m) rescaling as the single-GPU combine
("The Kernel Level: Attention and MoE", the split-KV section: split-KV with the
LSE merge is the DCP merge at another scale; "Attention at 128k", §2 for the
merge itself).

The step is graph-friendly: all ranks use one plan, made on the host for the
longest slice of each sequence, and read their own slice lengths from device
memory (decode_attn_splitk_dev), so the workspaces have the same layout on every
rank and the gathered buffer is the input of decode_attn_combine_ranks.

Slicing: rank r of R holds positions [r * L // R, (r + 1) * L // R) of a
sequence of length L; slices differ in length by at most one and are non-empty
when L >= R (required).

Several new tokens per sequence (q [B, q_len, Hq, Dk]): the new tokens are the
last q_len positions, so they fall in the last rank's slice (every slice must
hold at least q_len positions); that rank applies the causal limit among them
and every other rank, whose slice lies wholly before them, runs with
DA_FLAG_NO_CAUSAL.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import _native as N
from . import api as A


def context_slices(seq_lens: Sequence[int], world: int,
                   min_len: int = 1) -> List[Tuple[List[int], List[int]]]:
    """For every rank, (starts, lengths) of its slice of each sequence; every
    slice holds at least min_len positions."""
    if world < 1:
        raise ValueError("world must be >= 1")
    out = []
    for r in range(world):
        starts, lens = [], []
        for L in seq_lens:
            L = int(L)
            if L // world < min_len:
                raise ValueError(f"a sequence of length {L} cannot be split over {world} ranks "
                                 f"into slices of at least {min_len} positions")
            s, e = r * L // world, (r + 1) * L // world
            starts.append(s)
            lens.append(e - s)
        out.append((starts, lens))
    return out


def max_slice_lengths(seq_lens: Sequence[int], world: int) -> List[int]:
    """The longest slice of each sequence: what every rank's plan is made for."""
    return [-(-int(L) // world) for L in seq_lens]


def shard_cache(cache: torch.Tensor, seq_lens: Sequence[int], rank: int,
                world: int) -> torch.Tensor:
    """This rank's slices of a full cache [B, cap, Hkv, D], packed into a local
    cache [B, max_slice, Hkv, D] (positions past a slice are zero)."""
    starts, lens = context_slices(seq_lens, world)[rank]
    cap = max(max_slice_lengths(seq_lens, world))
    local = torch.zeros((cache.shape[0], cap) + tuple(cache.shape[2:]), dtype=cache.dtype,
                        device=cache.device)
    for b, (s, n) in enumerate(zip(starts, lens)):
        local[b, :n] = cache[b, s:s + n]
    return local


def gather(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather a rank's tensor into [world, *local.shape] (rank-major), the
    exchange step of a context-parallel decode. With no process group (a
    single rank) the local tensor is returned with a leading dimension of 1."""
    import torch.distributed as dist
    if group is None and not (dist.is_available() and dist.is_initialized()):
        return local.unsqueeze(0)
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(local.shape), dtype=local.dtype, device=local.device)
    if local.is_cuda:
        dist.all_gather_into_tensor(out.view(-1), local.contiguous().view(-1), group=group)
    else:
        dist.all_gather(list(out.unbind(0)), local.contiguous(), group=group)
    return out


class ContextParallelDecode:
    """One rank of a context-parallel decode step.

    q is the full query [B, Hq, Dk], or [B, q_len, Hq, Dk] for several new
    tokens (every rank has it); k_local / v_local are this rank's slices
    [B, max_slice, Hkv, D] (shard_cache). Calling the object runs the split
    kernel on the slice, gathers every rank's workspace and merges them into
    out (q's shape with Dv last) on every rank.
    """

    def __init__(self, q: torch.Tensor, k_local: torch.Tensor, v_local: torch.Tensor,
                 seq_lens: Sequence[int], scale: float, *, rank: int = 0, world: int = 1,
                 group=None, v_dim: Optional[int] = None,
                 out_dtype: torch.dtype = torch.float32):
        self.world, self.rank, self.group = world, rank, group
        self.q_len = q.shape[1] if q.dim() == 4 else 1
        flags = N.DA_FLAG_NO_COMBINE
        if self.q_len > 1 and rank < world - 1:
            flags |= N.DA_FLAG_NO_CAUSAL        # this slice lies before the new tokens
        self.args = A.make_args(q, k_local, v_local, scale, v_dim=v_dim, out_dtype=out_dtype,
                                flags=flags)
        self.plan = A.decode_attn_plan(self.args, max_slice_lengths(seq_lens, world))
        self.workspace = A.new_workspace(self.plan, device=q.device)
        _, lens = context_slices(seq_lens, world, self.q_len)[rank]
        self.local_lens = torch.tensor(lens, dtype=torch.int32, device=q.device)
        self.dev = A.make_dev(seq_lens=self.local_lens)

    def set_lengths(self, seq_lens: Sequence[int]) -> None:
        """New lengths (at most those of the plan's): only device memory changes,
        so a captured launch stays valid."""
        _, lens = context_slices(seq_lens, self.world, self.q_len)[self.rank]
        self.local_lens.copy_(torch.tensor(lens, dtype=torch.int32))

    def __call__(self, q: torch.Tensor, k_local: torch.Tensor, v_local: torch.Tensor,
                 out: torch.Tensor, stream=None) -> torch.Tensor:
        A.decode_attn_splitk_dev(self.args, self.plan, self.dev, q, k_local, v_local, out,
                                 self.workspace, stream)
        gathered = gather(self.workspace, self.group) if self.world > 1 else \
            self.workspace.unsqueeze(0)
        A.decode_attn_combine_ranks(self.args, self.plan, gathered, self.world, out, stream)
        return out
