"""Python binding of the C ABI, with the same names.

Argument marshalling only: tensors become device pointers and element
strides, the current torch stream becomes the cudaStream_t, and every
non-zero status becomes a DecodeAttnError carrying the library's message.
Every step of the computation runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from . import _native as N

_DT = {torch.float32: N.DA_F32, torch.float16: N.DA_F16, torch.bfloat16: N.DA_BF16}


class DecodeAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{N.STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


def _check(rc: int) -> None:
    if rc != N.DA_OK:
        raise DecodeAttnError(rc, decode_attn_last_error())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def dtype_code(dt: torch.dtype) -> int:
    if dt not in _DT:
        raise TypeError(f"unsupported dtype {dt}")
    return _DT[dt]


def make_args(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float, *,
              v_dim: Optional[int] = None, out_dtype: torch.dtype = torch.float32,
              force_splits: int = 0, flags: int = 0, timeout_us: int = 0) -> N.DaArgs:
    """Describe q [B, Hq, Dk] (one token per sequence) or [B, q_len, Hq, Dk]
    (q_len new tokens, causal among themselves) and caches [B, cap, Hkv, D]
    (any element strides) as a da_args_t. For MLA pass the same tensor as both
    caches and v_dim."""
    if q.dim() not in (3, 4) or k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, D] or [B, q_len, Hq, D] and caches [B, cap, Hkv, D]")
    if q.dim() == 3:
        (B, Hq, Dk), q_len = q.shape, 1
    else:
        B, q_len, Hq, Dk = q.shape
    a = N.DaArgs()
    a.batch, a.n_heads, a.n_kv_heads, a.head_dim = B, Hq, k_cache.shape[2], Dk
    a.q_len = q_len
    a.v_dim = int(v_dim) if v_dim is not None else v_cache.shape[3]
    a.capacity = k_cache.shape[1]
    ks, vs = k_cache.stride(), v_cache.stride()
    a.k_batch_stride, a.k_pos_stride, a.k_head_stride = ks[0], ks[1], ks[2]
    a.v_batch_stride, a.v_pos_stride, a.v_head_stride = vs[0], vs[1], vs[2]
    if ks[3] != 1 or vs[3] != 1:
        raise ValueError("the last cache dimension must be contiguous")
    a.kv_dtype = dtype_code(k_cache.dtype)
    a.out_dtype = dtype_code(out_dtype)
    a.scale = float(scale)
    a.force_splits = int(force_splits)
    a.flags = int(flags)
    a.timeout_us = int(timeout_us)
    return a


def decode_attn_plan(args: N.DaArgs, seq_lens_host: Sequence[int], num_sms: int = 0) -> N.DaPlan:
    lens = (ctypes.c_int32 * max(1, args.batch))(*[int(x) for x in seq_lens_host])
    plan = N.DaPlan()
    _check(N.load().decode_attn_plan(ctypes.byref(args), ctypes.cast(lens, ctypes.c_void_p),
                                     int(num_sms), ctypes.byref(plan)))
    return plan


def decode_attn_workspace_bytes(plan: N.DaPlan) -> int:
    return int(N.load().decode_attn_workspace_bytes(ctypes.byref(plan)))


def new_workspace(plan: N.DaPlan, device=None) -> torch.Tensor:
    """Caller-owned workspace for one device (torch's allocator aligns to 512 bytes)."""
    return torch.empty(decode_attn_workspace_bytes(plan), dtype=torch.uint8,
                       device=device or "cuda")


def decode_attn_splitk_ex(args: N.DaArgs, plan: N.DaPlan, q: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                          stream=None) -> None:
    _check(N.load().decode_attn_splitk_ex(ctypes.byref(args), ctypes.byref(plan), _ptr(q),
                                          _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(stream)))


def decode_attn_combine(args: N.DaArgs, plan: N.DaPlan, workspace: torch.Tensor,
                        out: torch.Tensor, stream=None) -> None:
    _check(N.load().decode_attn_combine(ctypes.byref(args), ctypes.byref(plan), _ptr(workspace),
                                        _ptr(out), _stream(stream)))


def decode_attn_combine_ranks(args: N.DaArgs, plan: N.DaPlan, workspaces: torch.Tensor,
                              n_ranks: int, out: torch.Tensor, stream=None) -> None:
    """Merge the partials of n_ranks ranks that ran the same plan on their slices
    of the context; `workspaces` holds their workspaces back to back."""
    _check(N.load().decode_attn_combine_ranks(ctypes.byref(args), ctypes.byref(plan),
                                              _ptr(workspaces), int(n_ranks), _ptr(out),
                                              _stream(stream)))


def decode_attn_splitk(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       seq_lens: Sequence[int], n_heads: int, n_kv_heads: int, head_dim: int,
                       scale: float, out: torch.Tensor, stream=None) -> None:
    """Short form: batch 1, f32 everything, caches [L, Hkv, D] contiguous."""
    lens = (ctypes.c_int32 * 1)(int(seq_lens[0]))
    _check(N.load().decode_attn_splitk(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       ctypes.cast(lens, ctypes.c_void_p), int(n_heads),
                                       int(n_kv_heads), int(head_dim), float(scale), _ptr(out),
                                       _stream(stream)))


def decode_attn_splitk_noalloc(args: N.DaArgs, plan: N.DaPlan, q: torch.Tensor,
                               k_cache: torch.Tensor, v_cache: torch.Tensor, out: torch.Tensor,
                               stream=None) -> None:
    """decode_attn_splitk_ex without a workspace: the partials go to a 16 MiB
    array inside the library (for callers that cannot allocate). Calls that
    overlap on the GPU share that array and race."""
    _check(N.load().decode_attn_splitk_noalloc(ctypes.byref(args), ctypes.byref(plan), _ptr(q),
                                               _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                               _stream(stream)))


def make_paged_args(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, scale: float,
                    max_blocks_per_seq: int, *, v_dim: Optional[int] = None,
                    out_dtype: torch.dtype = torch.float32, force_splits: int = 0,
                    flags: int = 0, timeout_us: int = 0) -> N.DaArgs:
    """da_args_t for paged pools [num_blocks, block_size, Hkv, D]: the position and
    head strides come from the pools, the capacity is max_blocks_per_seq *
    block_size (the batch strides are not used for addressing). For MLA pass the
    latent pool as both pools and v_dim."""
    if k_pool.dim() != 4 or v_pool.dim() != 4:
        raise ValueError("pools must be [num_blocks, block_size, Hkv, D]")
    a = make_args(q, k_pool, v_pool, scale, v_dim=v_dim, out_dtype=out_dtype,
                  force_splits=force_splits, flags=flags, timeout_us=timeout_us)
    a.capacity = int(max_blocks_per_seq) * k_pool.shape[1]
    return a


def make_dev(*, seq_lens: Optional[torch.Tensor] = None,
             block_table: Optional[torch.Tensor] = None, k_pool: Optional[torch.Tensor] = None,
             v_pool: Optional[torch.Tensor] = None) -> N.DaDev:
    """da_dev_t: device lengths (int32 [B] on the device) and, for paged caches, the
    block table (int32 [B, max_blocks] on the device) with the pools
    [num_blocks, block_size, Hkv, D]. The tensors must outlive every launch (and
    every replay of a captured launch) that uses them."""
    d = N.DaDev()
    if seq_lens is not None:
        if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda:
            raise TypeError("seq_lens must be an int32 CUDA tensor")
        d.seq_lens = seq_lens.data_ptr()
    if block_table is not None:
        if block_table.dtype != torch.int32 or not block_table.is_cuda or block_table.dim() != 2:
            raise TypeError("block_table must be a 2-D int32 CUDA tensor")
        if not block_table.is_contiguous():
            raise ValueError("block_table must be contiguous")
        if k_pool is None or v_pool is None:
            raise ValueError("a block table needs the K and V pools")
        d.block_table = block_table.data_ptr()
        d.max_blocks_per_seq = block_table.shape[1]
        d.block_size = k_pool.shape[1]
        d.num_blocks = k_pool.shape[0]
        d.k_block_stride = k_pool.stride(0)
        d.v_block_stride = v_pool.stride(0)
    return d


def decode_attn_splitk_dev(args: N.DaArgs, plan: N.DaPlan, dev: N.DaDev, q: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, out: torch.Tensor,
                           workspace: torch.Tensor, stream=None) -> None:
    """decode_attn_splitk_ex with lengths read on the device and, optionally,
    paged caches; capturable in a CUDA graph (no host decision depends on the
    current lengths)."""
    _check(N.load().decode_attn_splitk_dev(ctypes.byref(args), ctypes.byref(plan),
                                           ctypes.byref(dev), _ptr(q), _ptr(k_cache),
                                           _ptr(v_cache), _ptr(out), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(stream)))


def decode_attn_device_status(workspace: torch.Tensor, stream=None) -> None:
    _check(N.load().decode_attn_device_status(_ptr(workspace), _stream(stream)))


def decode_attn_last_error() -> str:
    return N.load().decode_attn_last_error().decode()


def decode_attn_release() -> None:
    N.load().decode_attn_release()


def decode_attn_version() -> str:
    return N.load().decode_attn_version().decode()


class DecodeAttention:
    """Plan once, run many times: holds the args, the plan and a workspace for
    fixed shapes and lengths (the plan/run split of the Kernel Level page)."""

    def __init__(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 seq_lens: Sequence[int], scale: Optional[float] = None, *,
                 v_dim: Optional[int] = None, out_dtype: torch.dtype = torch.float32,
                 force_splits: int = 0, flags: int = 0, num_sms: int = 0,
                 timeout_us: int = 0):
        sc = 1.0 / math.sqrt(q.shape[-1]) if scale is None else float(scale)
        self.args = make_args(q, k_cache, v_cache, sc, v_dim=v_dim, out_dtype=out_dtype,
                              force_splits=force_splits, flags=flags, timeout_us=timeout_us)
        self.plan = decode_attn_plan(self.args, list(seq_lens), num_sms)
        self.workspace = torch.empty(decode_attn_workspace_bytes(self.plan), dtype=torch.uint8,
                                     device=q.device)
        self.out_dtype = out_dtype

    def new_out(self, device) -> torch.Tensor:
        a = self.args
        shape = (a.batch, a.n_heads, a.v_dim) if a.q_len <= 1 else \
            (a.batch, a.q_len, a.n_heads, a.v_dim)
        return torch.empty(shape, dtype=self.out_dtype, device=device)

    def __call__(self, q, k_cache, v_cache, out=None, stream=None) -> torch.Tensor:
        if out is None:
            out = self.new_out(q.device)
        decode_attn_splitk_ex(self.args, self.plan, q, k_cache, v_cache, out, self.workspace,
                              stream)
        return out


def make_proj(w: torch.Tensor) -> N.DaProj:
    """da_proj_t for per-head projection weights w [n_heads, out_dim, v_dim]
    (f32 or bf16, on the device, last dimension contiguous). The tensor must
    outlive every launch that uses the descriptor."""
    if w.dim() != 3 or w.stride(2) != 1:
        raise ValueError("w must be [n_heads, out_dim, v_dim] with a contiguous last dimension")
    p = N.DaProj()
    p.w = w.data_ptr()
    p.w_dtype = dtype_code(w.dtype)
    p.out_dim = w.shape[1]
    p.head_stride, p.row_stride = w.stride(0), w.stride(1)
    return p


def decode_attn_combine_proj(args: N.DaArgs, plan: N.DaPlan, proj: N.DaProj,
                             workspaces: torch.Tensor, out: torch.Tensor, n_ranks: int = 1,
                             stream=None) -> None:
    """The merge of n_ranks workspaces (back to back) followed by the per-head
    projection: out [B, (q_len,) Hq, out_dim]."""
    _check(N.load().decode_attn_combine_proj(ctypes.byref(args), ctypes.byref(plan),
                                             ctypes.byref(proj), _ptr(workspaces),
                                             int(n_ranks), _ptr(out), _stream(stream)))


def decode_attn_splitk_proj(args: N.DaArgs, plan: N.DaPlan, proj: N.DaProj, q: torch.Tensor,
                            k_cache: torch.Tensor, v_cache: torch.Tensor, out: torch.Tensor,
                            workspace: torch.Tensor, stream=None) -> None:
    """Split kernel, then the combine fused with the per-head projection."""
    _check(N.load().decode_attn_splitk_proj(ctypes.byref(args), ctypes.byref(plan),
                                            ctypes.byref(proj), _ptr(q), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(out), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream)))
