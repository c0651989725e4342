"""GPU parity of context-parallel decode (DCP), with the ranks emulated on one
GPU: every rank's split kernel runs on its slice of the context with the shared
plan (decode_attn_splitk_dev, lengths on the device), the workspaces are placed
back to back as an all-gather would leave them, and decode_attn_combine_ranks
merges them. The result must match the oracle on the whole context ("The
Kernel Level: Attention and MoE", the split-KV/DCP section)."""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import dcp
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows

pytestmark = pytest.mark.gpu
_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def dcp_emulated(case, world, v_dim=None):
    lens = case.seq_lens.tolist()
    q = case.q.cuda()
    shared = case.shared_kv
    k_loc = [dcp.shard_cache(case.k, lens, r, world).cuda() for r in range(world)]
    v_loc = k_loc if shared else [dcp.shard_cache(case.v, lens, r, world).cuda()
                                  for r in range(world)]
    out_dt = _TDT[case.out_dtype]
    a = A.make_args(q, k_loc[0], v_loc[0], case.scale, v_dim=v_dim, out_dtype=out_dt,
                    flags=N.DA_FLAG_NO_COMBINE)
    p = A.decode_attn_plan(a, dcp.max_slice_lengths(lens, world))
    wsb = A.decode_attn_workspace_bytes(p)
    assert wsb % 256 == 0
    stacked = torch.full((world, wsb), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.empty(case.batch, case.n_heads, case.v_dim, dtype=out_dt, device="cuda")
    for r in range(world):
        _, local_lens = dcp.context_slices(lens, world)[r]
        d = A.make_dev(seq_lens=torch.tensor(local_lens, dtype=torch.int32, device="cuda"))
        A.decode_attn_splitk_dev(a, p, d, q, k_loc[r], v_loc[r], out, stacked[r])
    A.decode_attn_combine_ranks(a, p, stacked, world, out)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_gqa_context_parallel(world):
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[7001, 2999], kv_dtype="f16", scale=1 / 16, seed=700 + world)
    got = dcp_emulated(case, world)
    worst, rel = errors(case, got, oracle_rows(case))
    assert np.all(np.isfinite(got)) and worst <= TOL["f16"], (worst, rel)


def test_gqa_context_parallel_bf16_out_d128():
    case = W.make_case("t", batch=3, n_heads=32, n_kv_heads=8, head_dim=128,
                       seq_lens=[4000, 37, 9000], kv_dtype="bf16", out_dtype="bf16",
                       scale=1 / math.sqrt(128), seed=710)
    got = dcp_emulated(case, 3)
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL["bf16"], (worst, rel)


def test_mla_context_parallel():
    case = W.make_case("mla", batch=1, n_heads=96, n_kv_heads=1, head_dim=576, v_dim=512,
                       seq_lens=[16384], kv_dtype="f32", scale=1 / math.sqrt(576.0), seed=720,
                       std=0.5, shared_kv=True)
    got = dcp_emulated(case, 2, v_dim=512)
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= 2e-4, (worst, rel)


def test_single_rank_object_matches_the_plain_call():
    case = W.make_case("t", batch=2, n_heads=8, n_kv_heads=2, head_dim=256,
                       seq_lens=[3000, 1200], kv_dtype="f32", scale=1 / 16, seed=730)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    step = dcp.ContextParallelDecode(q, k, v, case.seq_lens.tolist(), case.scale)
    out = torch.empty(2, 8, 256, device="cuda")
    step(q, k, v, out)
    torch.cuda.synchronize()
    worst, rel = errors(case, out.double().cpu().numpy(), oracle_rows(case))
    assert worst <= TOL["f32"], (worst, rel)
    step.set_lengths([1500, 1200])            # shorter context, same plan and buffers
    step(q, k, v, out)
    torch.cuda.synchronize()
    short = W.make_case("t", batch=2, n_heads=8, n_kv_heads=2, head_dim=256,
                        seq_lens=[3000, 1200], kv_dtype="f32", scale=1 / 16, seed=730)
    import dataclasses
    short = dataclasses.replace(short, seq_lens=torch.tensor([1500, 1200], dtype=torch.int32))
    worst, rel = errors(short, out.double().cpu().numpy(), oracle_rows(short))
    assert worst <= TOL["f32"], (worst, rel)


@pytest.mark.parametrize("world", [2, 4])
def test_tensor_core_gqa_context_parallel(world):
    # 32 query heads over one KV head, f16: the tensor-core kernel on every rank
    case = W.make_case("t", batch=2, n_heads=32, n_kv_heads=1, head_dim=128,
                       seq_lens=[9001, 1234], kv_dtype="f16", seed=740 + world)
    got = dcp_emulated(case, world)
    worst, rel = errors(case, got, oracle_rows(case))
    assert np.all(np.isfinite(got)) and worst <= TOL["f16"], (worst, rel)


@pytest.mark.parametrize("shape,world", [("simt", 2), ("tc", 3), ("mla", 2), ("f32rows", 3)])
def test_context_parallel_several_new_tokens(shape, world):
    # the new tokens fall in the last rank's slice; the other ranks' slices lie
    # before them and run without the causal limit (DA_FLAG_NO_CAUSAL)
    import oracle
    if shape == "mla":
        case = W.make_case("mla", batch=1, n_heads=48, n_kv_heads=1, head_dim=576, v_dim=512,
                           seq_lens=[6000], kv_dtype="f32", scale=1 / math.sqrt(576.0),
                           seed=750, std=0.5, shared_kv=True)
        q_len, v_dim, bar = 2, 512, TOL["f32"]
    elif shape == "tc":
        case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                           seq_lens=[7001, 2999], kv_dtype="f16", scale=1 / 16, seed=751)
        q_len, v_dim, bar = 4, None, TOL["f16"]
    elif shape == "f32rows":   # 12 rows per KV head on an f32 cache: the f32 kernel
        case = W.make_case("t", batch=2, n_heads=24, n_kv_heads=4, head_dim=256,
                           seq_lens=[7001, 2999], kv_dtype="f32", scale=1 / 16, seed=754)
        q_len, v_dim, bar = 2, None, TOL["f32"]
    else:
        case = W.make_case("t", batch=2, n_heads=8, n_kv_heads=4, head_dim=256,
                           seq_lens=[7001, 2999], kv_dtype="f32", scale=1 / 16, seed=752)
        q_len, v_dim, bar = 2, None, TOL["f32"]
    lens = case.seq_lens.tolist()
    q4 = W.multi_token_q(case.batch, q_len, case.n_heads, case.head_dim, seed=753)
    q = q4.cuda()
    dv = case.v_dim
    wss, step = [], None
    for r in range(world):
        kl = dcp.shard_cache(case.k, lens, r, world).cuda()
        vl = kl if case.shared_kv else dcp.shard_cache(case.v, lens, r, world).cuda()
        step = dcp.ContextParallelDecode(q, kl, vl, lens, case.scale, rank=r, world=world,
                                         v_dim=v_dim)
        scratch = torch.empty(case.batch, q_len, case.n_heads, dv, device="cuda")
        A.decode_attn_splitk_dev(step.args, step.plan, step.dev, q, kl, vl, scratch,
                                 step.workspace)
        wss.append(step.workspace)
    out = torch.empty(case.batch, q_len, case.n_heads, dv, device="cuda")
    A.decode_attn_combine_ranks(step.args, step.plan, torch.stack(wss), world, out)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    ref = oracle.attention_multi(q4, case.k, case.v, case.seq_lens, case.scale, v_dim=dv,
                                 threads=0)
    worst = 0.0
    for b, L in enumerate(lens):
        for t in range(q_len):
            vm = float(case.v[b, :L - q_len + 1 + t, :, :dv].float().abs().max())
            worst = max(worst, float(np.max(np.abs(got[b, t] - ref[b, t]))) / vm)
    assert np.all(np.isfinite(got)) and worst <= bar, worst
