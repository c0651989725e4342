"""Decode-attention oracle (test infrastructure).

This package is TEST INFRASTRUCTURE. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The product library never loads it and shares no code with it.

``decode_attn_oracle.c`` holds the arithmetic (plain C, double precision,
optionally OpenMP over (batch, head) rows). This module only compiles it
with gcc, marshals arrays through ctypes and widens q to double.

What it computes: softmax(q K^T * scale) V for one query row per head,
head h reading KV head h // G (G = n_heads // n_kv_heads), attending to
positions 0 .. seq_lens[b]-1 of its batch element. That is the result the
split-KV method reaches exactly up to reassociation ("Attention at 128k:
Split Over Context, Split Over Heads", section 2; "The Kernel Level:
Attention and MoE", section "Decode Starves the SMs").

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(closed forms, brute force on tiny inputs, the split identity, the worked
merge example and planted-mistake negative controls).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liborc.so")

F32, F16, BF16, F64 = 0, 1, 2, 3
NC_NO_MERGE_RESCALE, NC_NO_ALPHA = 1, 2
MERGE_ML, MERGE_LSE = 0, 1

_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("v_dim", ctypes.c_int32), ("kv_type", ctypes.c_int32),
        ("k_batch_stride", ctypes.c_int64), ("k_pos_stride", ctypes.c_int64),
        ("k_head_stride", ctypes.c_int64),
        ("v_batch_stride", ctypes.c_int64), ("v_pos_stride", ctypes.c_int64),
        ("v_head_stride", ctypes.c_int64),
        ("scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP when available). Returns the .so path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_BUILD, exist_ok=True)
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler found")
    tmp = _LIB + f".{os.getpid()}.tmp"
    base = [cc, "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            L.orc_attention.argtypes = [ctypes.POINTER(_Shape), P, P, P, P, P, ctypes.c_int, P,
                                        ctypes.c_int]
            L.orc_attention.restype = ctypes.c_int
            L.orc_attention_split.argtypes = [ctypes.POINTER(_Shape), P, P, P, P, P, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, P, P, P, P]
            L.orc_attention_split.restype = ctypes.c_int
            L.orc_merge.argtypes = [ctypes.c_int, P, P, P, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, P, P, P]
            L.orc_merge.restype = ctypes.c_int
            L.orc_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def max_threads() -> int:
    return int(lib().orc_max_threads())


# ---------------------------------------------------------------------------
# array marshalling
# ---------------------------------------------------------------------------
def _storage(x):
    """(numpy array holding the stored bits, type tag, element strides) of a
    cache given as a numpy array or a CPU torch tensor of shape [B, cap, Hkv, D]."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.device.type != "cpu":
            raise ValueError("oracle inputs must be CPU tensors")
        if x.dtype == torch.bfloat16:
            arr, tag = x.view(torch.int16).numpy(), BF16
        elif x.dtype == torch.float16:
            arr, tag = x.numpy(), F16
        elif x.dtype == torch.float32:
            arr, tag = x.numpy(), F32
        elif x.dtype == torch.float64:
            arr, tag = x.numpy(), F64
        else:
            raise TypeError(f"unsupported cache dtype {x.dtype}")
    else:
        arr = np.asarray(x)
        tag = {np.dtype(np.float32): F32, np.dtype(np.float16): F16,
               np.dtype(np.float64): F64}.get(arr.dtype)
        if tag is None:
            raise TypeError(f"unsupported cache dtype {arr.dtype}")
    if arr.ndim != 4:
        raise ValueError("cache must be [batch, capacity, n_kv_heads, dim]")
    strides = tuple(s // arr.itemsize for s in arr.strides)
    return arr, tag, strides


def _prepare(q, k, v, seq_lens, scale, v_dim=None):
    q64 = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    if q64.ndim != 3:
        raise ValueError("q must be [batch, n_heads, head_dim]")
    ka, ktag, ks = _storage(k)
    va, vtag, vs = _storage(v)
    if ktag != vtag:
        raise TypeError("K and V must share a storage type")
    B, Hq, Dk = q64.shape
    if ka.shape[0] != B or ka.shape[3] < Dk:
        raise ValueError("K shape does not match q")
    Hkv = ka.shape[2]
    Dv = int(v_dim) if v_dim is not None else va.shape[3]
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(-1))
    if lens.shape[0] != B:
        raise ValueError("seq_lens must have one entry per batch element")
    if lens.min() < 1 or lens.max() > min(ka.shape[1], va.shape[1]):
        raise ValueError("seq_lens out of range")
    shp = _Shape(B, Hq, Hkv, Dk, Dv, ktag, ks[0], ks[1], ks[2], vs[0], vs[1], vs[2],
                 float(scale))
    return q64, ka, va, lens, shp


def _pairs_arg(pairs):
    if pairs is None:
        return None, 0
    p = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return p, p.shape[0]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, seq_lens, scale, *, v_dim=None, pairs=None, threads=1):
    """softmax(q K^T scale) V in double.

    q: [B, Hq, Dk] (any float type; widened exactly to double).
    k, v: [B, cap, Hkv, D] caches (numpy f32/f16/f64 or CPU torch incl. bf16);
      v may be the same buffer as k with v_dim < D (MLA: values are the first
      v_dim columns of each latent row).
    pairs: optional list of (b, h); then the result is [n_pairs, Dv].
    Returns float64 [B, Hq, Dv] (or [n_pairs, Dv]).
    """
    q64, ka, va, lens, shp = _prepare(q, k, v, seq_lens, scale, v_dim)
    p, n = _pairs_arg(pairs)
    rows = n if p is not None else shp.batch * shp.n_heads
    out = np.empty((rows, shp.v_dim), dtype=np.float64)
    rc = lib().orc_attention(ctypes.byref(shp), _ptr(q64), _ptr(ka), _ptr(va), _ptr(lens),
                             _ptr(p), n, _ptr(out), int(threads))
    if rc:
        raise ValueError("oracle rejected its arguments")
    return out if p is not None else out.reshape(shp.batch, shp.n_heads, shp.v_dim)


def attention_multi(q, k, v, seq_lens, scale, *, v_dim=None, pairs=None, threads=1):
    """Several new query tokens per sequence, causal among themselves, in double.

    q: [B, T, Hq, Dk]: the last T positions of each sequence, whose keys and
    values are already in the cache. Token t sits at position L - T + t and
    attends to positions 0 .. L - T + t, the causal mask of a decoder block
    ("Decoder Block 6: Online Attention, the Capstone", Lesson: each query row
    sees its own prefix), so token t is plain attention over a sequence of
    length L - T + t + 1 and the oracle forms it that way, token by token.
    Requires every seq_lens[b] >= T. Returns float64 [B, T, Hq, Dv] (with
    pairs (b, h): [T, n_pairs, Dv]).
    """
    q = q.detach().cpu() if hasattr(q, "detach") else np.asarray(q)
    T = int(q.shape[1])
    lens = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
    if T < 1 or np.any(lens < T):
        raise ValueError("every sequence needs at least q_len positions")
    outs = [attention(q[:, t], k, v, (lens - T + 1 + t).astype(np.int32), scale, v_dim=v_dim,
                      pairs=pairs, threads=threads) for t in range(T)]
    return np.stack(outs, axis=0 if pairs is not None else 1)


def attention_proj(q, k, v, seq_lens, scale, w, *, v_dim=None, pairs=None, threads=1):
    """Attention followed by a per-head output projection, in double:
    out[b][h][e] = sum_c W[h][e][c] * attn[b][h][c] (the MLA value up-projection
    wv_b applied to the merged latent, "Attention at 128k", §2: the output
    projection is a function of the merged result). q is [B, Hq, Dk] or
    [B, T, Hq, Dk] (attention_multi; every token of head h uses W[h]); w is
    [Hq, out_dim, v_dim] (numpy or CPU torch, any float type, widened exactly).
    With pairs (b, h) only those rows are formed: [n_pairs, out_dim] (or
    [T, n_pairs, out_dim])."""
    if hasattr(w, "detach"):                                # a CPU torch tensor (incl. bf16)
        import torch
        W = w.detach().cpu().to(torch.float64).numpy()
    else:
        W = np.asarray(w, dtype=np.float64)
    multi = len(q.shape) == 4
    att = (attention_multi if multi else attention)(q, k, v, seq_lens, scale, v_dim=v_dim,
                                                    pairs=pairs, threads=threads)
    if pairs is not None:
        Wp = W[[h for _, h in pairs]]                       # [n_pairs, out_dim, v_dim]
        return np.einsum("...pc,pec->...pe", att, Wp)
    return np.einsum("...hc,hec->...he", att, W)


def attention_split(q, k, v, seq_lens, scale, n_splits, *, block=64, form=MERGE_ML, flags=0,
                    v_dim=None, pairs=None, return_partials=False):
    """The split-KV method in double: n_splits contiguous segments per row, the
    online recurrence with block length `block` inside each, then the merge.
    With return_partials the per-segment (m, l, O) triples are returned too,
    shaped [rows, n_splits] and [rows, n_splits, Dv]."""
    q64, ka, va, lens, shp = _prepare(q, k, v, seq_lens, scale, v_dim)
    p, n = _pairs_arg(pairs)
    rows = n if p is not None else shp.batch * shp.n_heads
    out = np.empty((rows, shp.v_dim), dtype=np.float64)
    pm = pl = pO = None
    if return_partials:
        pm = np.empty((rows, n_splits), dtype=np.float64)
        pl = np.empty((rows, n_splits), dtype=np.float64)
        pO = np.empty((rows, n_splits, shp.v_dim), dtype=np.float64)
    rc = lib().orc_attention_split(ctypes.byref(shp), _ptr(q64), _ptr(ka), _ptr(va), _ptr(lens),
                                   _ptr(p), n, int(n_splits), int(block), int(form), int(flags),
                                   _ptr(out), _ptr(pm), _ptr(pl), _ptr(pO))
    if rc:
        raise ValueError("oracle rejected its arguments")
    if p is None:
        out = out.reshape(shp.batch, shp.n_heads, shp.v_dim)
    return (out, pm, pl, pO) if return_partials else out


def merge(m, l, O, *, form=MERGE_ML, flags=0):
    """Merge partial triples: m, l [n], O [n, dv] (un-normalised).
    Returns (m_merged, l_merged, out[dv])."""
    m = np.ascontiguousarray(np.asarray(m, dtype=np.float64).reshape(-1))
    l = np.ascontiguousarray(np.asarray(l, dtype=np.float64).reshape(-1))
    O = np.ascontiguousarray(np.asarray(O, dtype=np.float64).reshape(m.shape[0], -1))
    dv = O.shape[1]
    out = np.empty(dv, dtype=np.float64)
    mo, lo = ctypes.c_double(), ctypes.c_double()
    rc = lib().orc_merge(m.shape[0], _ptr(m), _ptr(l), _ptr(O), dv, int(form), int(flags),
                         ctypes.cast(ctypes.byref(mo), ctypes.c_void_p),
                         ctypes.cast(ctypes.byref(lo), ctypes.c_void_p), _ptr(out))
    if rc:
        raise ValueError("merge of only empty partials is undefined")
    return mo.value, lo.value, out
