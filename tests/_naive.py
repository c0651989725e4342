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


def naive_causal_attention(q, k, v, seq_lens, scale, v_dim=None) -> np.ndarray:
    """q [B, T, Hq, Dk]: the last T positions of each sequence. One materialised
    [T*G, L] score matrix per (sequence, KV head) with an explicit causal mask
    (query row of token t may see key j iff j <= L - T + t), softmax, times V."""
    Q = widen(q)
    K = widen(k)
    V = widen(v)
    B, T, Hq, Dk = Q.shape
    Hkv = K.shape[2]
    G = Hq // Hkv
    Dv = V.shape[3] if v_dim is None else int(v_dim)
    out = np.zeros((B, T, Hq, Dv))
    for b in range(B):
        L = int(seq_lens[b])
        j = np.arange(L)
        for g in range(Hkv):
            Qg = Q[b, :, g * G:(g + 1) * G, :].reshape(T * G, Dk)       # rows (t, head)
            S = (Qg @ K[b, :L, g, :Dk].T) * scale                      # [T*G, L]
            tok = np.repeat(np.arange(T), G)
            mask = j[None, :] <= (L - T + tok)[:, None]
            S = np.where(mask, S, -np.inf)
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P = P / P.sum(axis=1, keepdims=True)
            out[b, :, g * G:(g + 1) * G, :] = (P @ V[b, :L, g, :Dv]).reshape(T, G, Dv)
    return out
