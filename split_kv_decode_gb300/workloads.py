"""Seeded synthetic inputs for decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, and it imports neither the CUDA binding nor the oracle.
The tests, the smoke check and the benchmark use it to give both sides the
same bits.

Every case draws from a CPU ``torch.Generator`` seeded explicitly, in a fixed
order: q first, then for each batch element its K rows, then its V rows. K/V
are drawn in float32 and rounded once to the storage type, so the stored
values are the values both sides read. Positions past a sequence's length
(up to the cache capacity) are filled with NaN, so any read of them that is
not masked shows up in the output.

The named cases follow the geometries the pages work with:
  * ``gqa_8x2``    8 query / 2 KV heads, head_dim 256, f32 KV, L = 4096
  * ``gqa_16x4``   16 / 4 heads (G = 4), head_dim 256, f16 KV, f32 q; the
                   rungs 4096 / 20480 / 61440 / 151552 / 262144
                   (aprender issue 3725 design note, §1 geometry and §4 rungs)
  * ``mla_96``     96 query heads over one shared 576-wide latent row per
                   position (512 latent + 64 rope), values = first 512
                   columns, f32 cache N(0, 0.5), L = 131072, about 302 MB
                   ("Attention at 128k", §1.1)
  * ``gqa_24x4``   24 / 4 heads (G = 6), head_dim 256, f32 KV, batch 4 with
                   lengths 8192 / 20480 / 61440 / 131072
  * ``ragged_32``  batch 32, 32 / 8 heads, head_dim 128, bf16 KV, lengths
                   uniform in [1024, 131072] from the seed, bf16 output
Two MLA variants the pages name beside the 96-head f32 cache:
  * ``mla_128``    128 heads over the same latent ("The Kernel Level", absorbed
                   MLA decode: one latent for 128 heads)
  * ``mla_96_f16`` 96 heads over an f16 latent cache ("Attention at 128k" §1:
                   the reference engine's compressed cache is f16)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

F32, F16, BF16 = "f32", "f16", "bf16"
_TORCH = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}


@dataclasses.dataclass
class Case:
    name: str
    batch: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    v_dim: int
    seq_lens: torch.Tensor          # int32 [B], CPU
    capacity: int
    kv_dtype: str
    out_dtype: str
    scale: float
    q: torch.Tensor                 # f32 [B, Hq, Dk], CPU
    k: torch.Tensor                 # [B, cap, Hkv, Dk] storage dtype, CPU
    v: torch.Tensor                 # [B, cap, Hkv, Dv_storage]; for MLA the same tensor as k
    shared_kv: bool = False         # MLA: values are the first v_dim columns of k

    @property
    def kv_bytes(self) -> int:
        """K+V bytes that must be read once per decode step (for MLA the value
        columns are a prefix of the key row and count once)."""
        es = torch.empty((), dtype=_TORCH[self.kv_dtype]).element_size()
        L = int(self.seq_lens.sum())
        if self.shared_kv:
            return L * self.n_kv_heads * self.head_dim * es
        return L * self.n_kv_heads * (self.head_dim + self.v_dim) * es


def _draw(gen: torch.Generator, shape, std: float, dtype: str) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=gen.device)
    if std != 1.0:
        x.mul_(std)
    return x.to(_TORCH[dtype])


def make_case(name: str, *, batch: int, n_heads: int, n_kv_heads: int, head_dim: int,
              seq_lens: Sequence[int], kv_dtype: str = F32, out_dtype: str = F32,
              v_dim: Optional[int] = None, scale: Optional[float] = None, seed: int = 1234,
              std: float = 1.0, shared_kv: bool = False, capacity: Optional[int] = None,
              q_zero: bool = False, poison_tail: bool = True, device: str = "cpu") -> Case:
    """Draw one seeded case. ``shared_kv`` builds an MLA-style cache where the
    values are the first ``v_dim`` columns of each key row. With a CUDA
    ``device`` the same recipe is drawn there from a generator of that device
    (other values of the same distributions, for timing large workloads
    without a host round trip; parity checks use CPU draws)."""
    lens = torch.tensor(list(seq_lens), dtype=torch.int32)
    assert lens.numel() == batch and int(lens.min()) >= 1
    cap = int(capacity) if capacity is not None else int(lens.max())
    assert cap >= int(lens.max())
    dv = head_dim if v_dim is None else int(v_dim)
    sc = 1.0 / math.sqrt(head_dim) if scale is None else float(scale)
    g = torch.Generator(device=device).manual_seed(int(seed))
    q = torch.randn((batch, n_heads, head_dim), generator=g, dtype=torch.float32, device=device)
    if q_zero:
        q.zero_()
    tdt = _TORCH[kv_dtype]
    k = torch.empty((batch, cap, n_kv_heads, head_dim), dtype=tdt, device=device)
    v = k if shared_kv else torch.empty((batch, cap, n_kv_heads, dv), dtype=tdt, device=device)
    for b in range(batch):
        L = int(lens[b])
        k[b, :L] = _draw(g, (L, n_kv_heads, head_dim), std, kv_dtype)
        if not shared_kv:
            v[b, :L] = _draw(g, (L, n_kv_heads, dv), std, kv_dtype)
        if L < cap:
            fill = float("nan") if poison_tail else 0.0
            k[b, L:] = fill
            if not shared_kv:
                v[b, L:] = fill
    return Case(name, batch, n_heads, n_kv_heads, head_dim, dv, lens, cap, kv_dtype,
                out_dtype, sc, q, k, v, shared_kv)


def multi_token_q(batch: int, q_len: int, n_heads: int, head_dim: int, seed: int = 4321,
                  std: float = 1.0) -> torch.Tensor:
    """Seeded f32 queries [B, q_len, Hq, Dk] for q_len new tokens per sequence
    (their keys and values are the last q_len rows of each cache)."""
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((batch, q_len, n_heads, head_dim), generator=g, dtype=torch.float32)
    return q.mul_(std) if std != 1.0 else q


GQA16X4_RUNGS = (4096, 20480, 61440, 151552, 262144)
GQA24X4_LENS = (8192, 20480, 61440, 131072)


def ragged_lens(seed: int, batch: int = 32, lo: int = 1024, hi: int = 131072):
    """Sequence lengths drawn uniform in [lo, hi] from their own seeded generator."""
    g = torch.Generator().manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]


def named(name: str, *, seed: Optional[int] = None, seq_len: Optional[int] = None,
          scale_lens: float = 1.0, device: str = "cpu") -> Case:
    """The named workloads. ``seq_len`` overrides the context of a batch-1 case;
    ``scale_lens`` shrinks every length (for quick, oracle-sized variants);
    ``device`` draws on that device (see make_case)."""
    def L(x):
        return max(1, int(round(x * scale_lens)))

    def mk(*a, **kw):
        return make_case(*a, device=device, **kw)

    if name == "gqa_8x2":
        s = 1234 if seed is None else seed
        return mk(name, batch=1, n_heads=8, n_kv_heads=2, head_dim=256,
                  seq_lens=[L(seq_len or 4096)], kv_dtype=F32, scale=1.0 / 16, seed=s)
    if name == "gqa_16x4":
        s = 1235 if seed is None else seed
        return mk(name, batch=1, n_heads=16, n_kv_heads=4, head_dim=256,
                  seq_lens=[L(seq_len or 151552)], kv_dtype=F16, scale=1.0 / 16, seed=s)
    if name == "mla_96":
        s = 1236 if seed is None else seed
        return mk(name, batch=1, n_heads=96, n_kv_heads=1, head_dim=576, v_dim=512,
                  seq_lens=[L(seq_len or 131072)], kv_dtype=F32,
                  scale=1.0 / math.sqrt(576.0), seed=s, std=0.5, shared_kv=True)
    if name == "mla_128":   # the absorbed MLA shape with 128 heads ("The Kernel Level")
        s = 1239 if seed is None else seed
        return mk(name, batch=1, n_heads=128, n_kv_heads=1, head_dim=576, v_dim=512,
                  seq_lens=[L(seq_len or 131072)], kv_dtype=F32,
                  scale=1.0 / math.sqrt(576.0), seed=s, std=0.5, shared_kv=True)
    if name == "mla_96_f16":  # the compressed cache in f16 ("Attention at 128k", §1)
        s = 1240 if seed is None else seed
        return mk(name, batch=1, n_heads=96, n_kv_heads=1, head_dim=576, v_dim=512,
                  seq_lens=[L(seq_len or 131072)], kv_dtype=F16,
                  scale=1.0 / math.sqrt(576.0), seed=s, std=0.5, shared_kv=True)
    if name == "gqa_24x4":
        s = 1237 if seed is None else seed
        return mk(name, batch=4, n_heads=24, n_kv_heads=4, head_dim=256,
                  seq_lens=[L(x) for x in GQA24X4_LENS], kv_dtype=F32,
                  scale=1.0 / 16, seed=s)
    if name == "ragged_32":
        s = 1238 if seed is None else seed
        lens = [L(x) for x in ragged_lens(s)]
        return mk(name, batch=32, n_heads=32, n_kv_heads=8, head_dim=128,
                  seq_lens=lens, kv_dtype=BF16, out_dtype=BF16,
                  scale=1.0 / math.sqrt(128.0), seed=s)
    raise KeyError(name)


NAMES = ("gqa_8x2", "gqa_16x4", "mla_96", "gqa_24x4", "ragged_32", "mla_128", "mla_96_f16")
