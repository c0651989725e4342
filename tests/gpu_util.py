"""Helpers for the GPU parity tests: run a seeded case through the C ABI and
compare it with the oracle.

Error metric (the tolerance the parity bar states): for every (b, h) row,
max_e |gpu - oracle| divided by max |V| over the rows that (b) attends to;
the reported error is the maximum over rows. relL2 against the oracle's
output norm is reported as well, as the sharper diagnostic.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W

TOL = {"f32": 2e-4, "f16": 5e-3, "bf16": 5e-3}
_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_device(case: W.Case, device="cuda"):
    q = case.q.to(device)
    k = case.k.to(device)
    v = k if case.shared_kv else case.v.to(device)
    return q, k, v


def run(case: W.Case, *, dev=None, force_splits=0, flags=0, num_sms=0, poison_ws=False,
        timeout_us=0):
    """Run the case through DecodeAttention (plan + decode_attn_splitk_ex).
    Returns (out as float64 numpy [B, Hq, Dv], the DecodeAttention object)."""
    q, k, v = dev if dev is not None else to_device(case)
    da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale, v_dim=case.v_dim,
                           out_dtype=_TDT[case.out_dtype], force_splits=force_splits,
                           flags=flags, num_sms=num_sms, timeout_us=timeout_us)
    if poison_ws:
        da.workspace.fill_(0xFF)            # every float in it reads as NaN
    out = da(q, k, v)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    return out.double().cpu().numpy(), da


def oracle_rows(case: W.Case, pairs=None, threads=0):
    return oracle.attention(case.q, case.k, case.v, case.seq_lens, case.scale,
                            v_dim=case.v_dim, pairs=pairs, threads=threads)


def vmax_per_batch(case: W.Case):
    out = []
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        x = case.v[b, :L, :, :case.v_dim].float()
        out.append(float(x.abs().max()))
    return out


def errors(case: W.Case, got: np.ndarray, ref: np.ndarray, pairs=None):
    """(max |err| / max|V| over rows, relL2) for got vs ref. got is [B, Hq, Dv];
    ref is [B, Hq, Dv] or, with pairs, [n_pairs, Dv]."""
    vm = vmax_per_batch(case)
    if pairs is None:
        pairs = [(b, h) for b in range(case.batch) for h in range(case.n_heads)]
        ref = ref.reshape(-1, ref.shape[-1])
    g = np.stack([got[b, h] for b, h in pairs])
    worst = max(float(np.max(np.abs(g[i] - ref[i]))) / vm[b] for i, (b, _) in enumerate(pairs))
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300))
    return worst, rel


def sample_pairs(case: W.Case, per_batch=2, seed=0):
    rng = np.random.default_rng(seed)
    pairs = []
    for b in range(case.batch):
        hs = sorted(rng.choice(case.n_heads, size=min(per_batch, case.n_heads), replace=False))
        pairs += [(b, int(h)) for h in hs]
    return pairs
