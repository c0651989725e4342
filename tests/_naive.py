"""Brute-force materialised attention in numpy float64, used only to pin the oracle.

This is the "naive attention" formulation of "The Kernel Level: Attention and
MoE" (section "Naive Attention"): build the whole score matrix S = Q K^T for a
KV head's group of query heads, softmax every row, multiply by V. It shares
nothing with the C oracle (different language, different loop order, library
matmul, widening done by numpy/torch instead of the oracle's bit decoders), so
agreement between the two on tiny inputs pins the oracle's indexing, grouping
and masking.
"""
from __future__ import annotations

import numpy as np
import torch


def widen(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def naive_attention(q, k, v, seq_lens, scale, v_dim=None) -> np.ndarray:
    Q = widen(q)
    K = widen(k)
    V = widen(v)
    B, Hq, Dk = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    Dv = V.shape[3] if v_dim is None else int(v_dim)
    out = np.zeros((B, Hq, Dv))
    for b in range(B):
        L = int(seq_lens[b])
        for g in range(Hkv):
            Qg = Q[b, g * G:(g + 1) * G, :]                 # [G, Dk]
            S = (Qg @ K[b, :L, g, :Dk].T) * scale            # [G, L], materialised
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P = P / P.sum(axis=1, keepdims=True)             # softmax rows
            out[b, g * G:(g + 1) * G, :] = P @ V[b, :L, g, :Dv]
    return out
