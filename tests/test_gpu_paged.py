"""GPU parity of decode_attn_splitk_dev: lengths read on the device, paged K/V
caches behind a block table, and a launch captured in a CUDA graph and replayed
while the contexts grow ("The Kernel Level: Attention and MoE", the serving and
CUDA-graph sections). Every result is compared with the oracle on the lengths
the launch attends over; the pages' storage layout plays no part in the oracle,
which reads the same values gathered back into a contiguous cache."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, to_device

pytestmark = pytest.mark.gpu

_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def at_lengths(case, lens):
    """The same case attending over other lengths (the cache is unchanged)."""
    return dataclasses.replace(case, seq_lens=torch.tensor(lens, dtype=torch.int32))


def paged(case, block_size, seed=0, spare=5):
    """Scatter the contiguous caches [B, cap, Hkv, D] into pools
    [num_blocks, block_size, Hkv, D] in a random block order. Unused pool blocks
    (and unused table entries, which point at them) hold NaN."""
    B, cap, hkv, d = case.k.shape
    nb_seq = -(-cap // block_size)
    num_blocks = B * nb_seq + spare
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(num_blocks, generator=g)
    kp = torch.full((num_blocks, block_size, hkv, d), float("nan"), dtype=case.k.dtype)
    vp = torch.full((num_blocks, block_size, hkv, case.v.shape[3]), float("nan"),
                    dtype=case.v.dtype)
    table = torch.full((B, nb_seq + 2), int(order[-1]), dtype=torch.int32)
    i = 0
    for b in range(B):
        for j in range(nb_seq):
            blk = int(order[i])
            i += 1
            n = min(block_size, cap - j * block_size)
            kp[blk, :n] = case.k[b, j * block_size:j * block_size + n]
            vp[blk, :n] = case.v[b, j * block_size:j * block_size + n]
            table[b, j] = blk
    return kp, vp, table


def run_dev(case, lens_now, *, kp=None, vp=None, table=None, flags=0):
    """Plan for case.seq_lens, attend over lens_now (read on the device)."""
    q = case.q.cuda()
    out_dt = _TDT[case.out_dtype]
    if table is None:
        _, k, v = to_device(case)
        a = A.make_args(q, k, v, case.scale, out_dtype=out_dt, flags=flags)
        dev_lens = torch.tensor(lens_now, dtype=torch.int32, device="cuda")
        d = A.make_dev(seq_lens=dev_lens)
    else:
        k, v = kp.cuda(), vp.cuda()
        tab = table.cuda()
        a = A.make_paged_args(q, k, v, case.scale, tab.shape[1], out_dtype=out_dt, flags=flags)
        dev_lens = torch.tensor(lens_now, dtype=torch.int32, device="cuda")
        d = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=v)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    ws.fill_(0xFF)                        # poisoned: every partial must be written
    out = torch.empty(case.batch, case.n_heads, case.v_dim, dtype=out_dt, device="cuda")
    A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    return out.double().cpu().numpy()


def check_against_oracle(case, lens_now, got):
    ref_case = at_lengths(case, lens_now)
    worst, rel = errors(ref_case, got, oracle_rows(ref_case))
    assert np.all(np.isfinite(got))
    assert worst <= TOL[case.kv_dtype], (worst, rel)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_device_lengths_shorter_than_the_plan(dtype):
    case = W.make_case("t", batch=3, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[5000, 3001, 700], kv_dtype=dtype, scale=1 / 16, seed=601)
    lens_now = [4000, 1, 700]
    check_against_oracle(case, lens_now, run_dev(case, lens_now))


def test_device_lengths_are_kept_within_one_and_the_plan():
    case = W.make_case("t", batch=2, n_heads=8, n_kv_heads=2, head_dim=128,
                       seq_lens=[2000, 900], kv_dtype="bf16", seed=602)
    got = run_dev(case, [0, 100000])          # -> [1, 900]
    check_against_oracle(case, [1, 900], got)


def test_device_lengths_equal_to_the_plan_match_the_plain_call_bit_for_bit():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[6000, 2500], kv_dtype="f16", scale=1 / 16, seed=603)
    got = run_dev(case, [6000, 2500])
    q, k, v = to_device(case)
    a = A.make_args(q, k, v, case.scale)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    out = torch.empty(2, 16, 256, device="cuda")
    A.decode_attn_splitk_ex(a, p, q, k, v, out, ws)
    assert np.array_equal(got, out.double().cpu().numpy())


@pytest.mark.parametrize("block_size", [16, 64, 256])
@pytest.mark.parametrize("geom", [(16, 4, 256, "f16"), (32, 8, 128, "bf16"), (8, 2, 256, "f32"),
                                  (48, 8, 128, "f16")])
def test_paged_cache(block_size, geom):
    hq, hkv, d, dtype = geom
    case = W.make_case("t", batch=3, n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=[3000, 1, 1207], kv_dtype=dtype, scale=1 / math.sqrt(d),
                       seed=610 + block_size + hq)
    kp, vp, table = paged(case, block_size, seed=block_size)
    got = run_dev(case, case.seq_lens.tolist(), kp=kp, vp=vp, table=table)
    check_against_oracle(case, case.seq_lens.tolist(), got)


def test_paged_cache_with_device_lengths_and_forced_splits():
    case = W.make_case("t", batch=2, n_heads=32, n_kv_heads=8, head_dim=128,
                       seq_lens=[9000, 4100], kv_dtype="bf16", out_dtype="bf16", seed=620)
    kp, vp, table = paged(case, 32, seed=3)
    q = case.q.cuda()
    k, v, tab = kp.cuda(), vp.cuda(), table.cuda()
    for lens_now, force in (([9000, 4100], 0), ([5333, 17], 0), ([9000, 4100], 7)):
        a = A.make_paged_args(q, k, v, case.scale, tab.shape[1], out_dtype=torch.bfloat16,
                              force_splits=force)
        dev_lens = torch.tensor(lens_now, dtype=torch.int32, device="cuda")
        d = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=v)
        p = A.decode_attn_plan(a, case.seq_lens.tolist())
        ws = A.new_workspace(p)
        out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device="cuda")
        A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws)
        torch.cuda.synchronize()
        check_against_oracle(case, lens_now, out.double().cpu().numpy())


def test_paged_decode_steps_replayed_from_one_cuda_graph():
    """A decode loop: the plan and the launch are captured once for the largest
    lengths; every step appends a K/V row to each sequence's pages, moves the
    device lengths on by one and replays the graph."""
    final = [3500, 2100, 901]
    case = W.make_case("t", batch=3, n_heads=16, n_kv_heads=4, head_dim=256, seq_lens=final,
                       kv_dtype="f16", scale=1 / 16, seed=630)
    bs = 64
    kp, vp, table = paged(case, bs, seed=9)
    q = case.q.cuda()
    k, v, tab = kp.cuda(), vp.cuda(), table.cuda()
    a = A.make_paged_args(q, k, v, case.scale, tab.shape[1])
    p = A.decode_attn_plan(a, final)
    ws = A.new_workspace(p)
    out = torch.empty(3, 16, 256, device="cuda")
    start = [f - 6 for f in final]
    dev_lens = torch.tensor(start, dtype=torch.int32, device="cuda")
    d = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=v)
    # positions >= the current length hold garbage until "written" by a step
    for b, L0 in enumerate(start):
        for pos in range(L0, final[b]):
            blk, slot = int(table[b, pos // bs]), pos % bs
            k[blk, slot] = float("nan")
            v[blk, slot] = float("nan")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):          # warm-up outside the capture
        A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, stream)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, stream)
    lens = list(start)
    for step in range(7):
        if step > 0:                         # append one row per sequence, then replay
            for b in range(3):
                pos = lens[b]
                blk, slot = int(table[b, pos // bs]), pos % bs
                k[blk, slot] = case.k[b, pos].cuda()
                v[blk, slot] = case.v[b, pos].cuda()
                lens[b] += 1
            dev_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        check_against_oracle(case, lens, out.double().cpu().numpy())
    assert lens == final


# ---------------------------------------------------------------------------
# MLA: one latent pool (values are the first 512 columns of each row)
# ---------------------------------------------------------------------------
MLA_F32_BAR = 2e-4   # f32 latent cache: the f32 bar at every length


def mla_case(lens, seed):
    return W.make_case("mla", batch=len(lens), n_heads=96, n_kv_heads=1, head_dim=576,
                       v_dim=512, seq_lens=lens, kv_dtype="f32", scale=1 / math.sqrt(576.0),
                       seed=seed, std=0.5, shared_kv=True)


def mla_pool(case, block_size, seed):
    B, cap = case.k.shape[:2]
    nb_seq = -(-cap // block_size)
    num_blocks = B * nb_seq + 3
    order = torch.randperm(num_blocks, generator=torch.Generator().manual_seed(seed))
    pool = torch.full((num_blocks, block_size, 1, 576), float("nan"))
    table = torch.full((B, nb_seq + 1), int(order[-1]), dtype=torch.int32)
    i = 0
    for b in range(B):
        for j in range(nb_seq):
            blk = int(order[i])
            i += 1
            n = min(block_size, cap - j * block_size)
            pool[blk, :n] = case.k[b, j * block_size:j * block_size + n]
            table[b, j] = blk
    return pool, table


def run_mla_dev(case, lens_now, pool=None, table=None):
    q = case.q.cuda()
    dev_lens = torch.tensor(lens_now, dtype=torch.int32, device="cuda")
    if pool is None:
        k = case.k.cuda()
        a = A.make_args(q, k, k, case.scale, v_dim=512)
        d = A.make_dev(seq_lens=dev_lens)
    else:
        k, tab = pool.cuda(), table.cuda()
        a = A.make_paged_args(q, k, k, case.scale, tab.shape[1], v_dim=512)
        d = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=k)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    assert p.kernel == N.DA_KERNEL_MLA_TC
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.empty(case.batch, 96, 512, device="cuda")
    A.decode_attn_splitk_dev(a, p, d, q, k, k, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    return out.double().cpu().numpy()


def check_mla(case, lens_now, got):
    ref_case = at_lengths(case, lens_now)
    worst, rel = errors(ref_case, got, oracle_rows(ref_case))
    bar = MLA_F32_BAR
    assert np.all(np.isfinite(got))
    assert worst <= bar, (worst, rel)


def test_mla_device_lengths_leave_empty_splits_neutral():
    case = mla_case([12000, 5000], seed=640)
    # the plan cuts 12000 positions into many splits; at 4500 most of them are empty
    for lens_now in ([4500, 5000], [12000, 4096], [1, 5000]):
        check_mla(case, lens_now, run_mla_dev(case, lens_now))


@pytest.mark.parametrize("block_size", [16, 64, 128])
def test_mla_paged_latent_pool(block_size):
    case = mla_case([6000, 4500], seed=650 + block_size)
    pool, table = mla_pool(case, block_size, seed=block_size)
    check_mla(case, [6000, 4500], run_mla_dev(case, [6000, 4500], pool, table))
    check_mla(case, [4200, 4096], run_mla_dev(case, [4200, 4096], pool, table))


def test_mla_paged_launch_replayed_from_a_cuda_graph():
    case = mla_case([8000], seed=660)
    pool, table = mla_pool(case, 64, seed=1)
    q = case.q.cuda()
    k, tab = pool.cuda(), table.cuda()
    a = A.make_paged_args(q, k, k, case.scale, tab.shape[1], v_dim=512)
    p = A.decode_attn_plan(a, [8000])
    ws = A.new_workspace(p)
    out = torch.empty(1, 96, 512, device="cuda")
    dev_lens = torch.tensor([5000], dtype=torch.int32, device="cuda")
    d = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=k)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        A.decode_attn_splitk_dev(a, p, d, q, k, k, out, ws, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.decode_attn_splitk_dev(a, p, d, q, k, k, out, ws, s)
    for L in (5000, 6500, 8000, 4096):
        dev_lens.fill_(L)
        g.replay()
        torch.cuda.synchronize()
        check_mla(case, [L], out.double().cpu().numpy())
