"""Host-side tests of the multi-rank paths, run as world-size-2 and -3 gloo
process groups on CPU (127.0.0.1):

* context-parallel decode (DCP): each rank takes its slice of every sequence
  (split_kv_decode_gb300.dcp), forms the slice's partial (m, l, acc) -- here with
  the oracle, standing in for the split kernel, which needs a GPU -- the ranks
  exchange them with dcp.gather, and the merge of all ranks' partials equals
  attention over the whole context ("The Kernel Level: Attention and MoE", the
  split-KV/DCP section);
* the bench's timing: the job's time is the slowest rank's (max over ranks).
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from split_kv_decode_gb300 import dcp
from split_kv_decode_gb300 import workloads as W


def test_context_slices_partition_every_sequence():
    lens = [7, 100, 4097, 3]
    for world in (1, 2, 3):
        sl = dcp.context_slices(lens, world)
        mx = dcp.max_slice_lengths(lens, world)
        for b, L in enumerate(lens):
            covered = []
            for r in range(world):
                s, n = sl[r][0][b], sl[r][1][b]
                assert 1 <= n <= mx[b] and n >= L // world
                covered += list(range(s, s + n))
            assert covered == list(range(L))            # contiguous, in rank order
    with pytest.raises(ValueError):
        dcp.context_slices([3], 4)


def test_shard_cache_packs_each_slice_at_position_zero():
    case = W.make_case("t", batch=2, n_heads=4, n_kv_heads=2, head_dim=16, seq_lens=[9, 5],
                       seed=7)
    for r in range(2):
        local = dcp.shard_cache(case.k, [9, 5], r, 2)
        starts, lens = dcp.context_slices([9, 5], 2)[r]
        assert local.shape[1] == 5
        for b in range(2):
            assert torch.equal(local[b, :lens[b]], case.k[b, starts[b]:starts[b] + lens[b]])
            assert torch.count_nonzero(local[b, lens[b]:]) == 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _dcp_rank(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lens = [301, 64, 1000]
        case = W.make_case("t", batch=3, n_heads=8, n_kv_heads=2, head_dim=32, seq_lens=lens,
                           kv_dtype="f16", seed=77)
        _, local_lens = dcp.context_slices(lens, world)[rank]
        k = dcp.shard_cache(case.k, lens, rank, world)
        v = dcp.shard_cache(case.v, lens, rank, world)
        # this rank's partial over its slice (one segment per row), in double
        _, m, l, O = oracle.attention_split(case.q, k, v, torch.tensor(local_lens), case.scale,
                                            1, return_partials=True)
        mine = torch.from_numpy(np.concatenate([m, l, O[:, 0, :]], axis=1))
        got = dcp.gather(mine)                               # [world, rows, 2 + dv]
        assert got.shape == (world,) + tuple(mine.shape)
        assert torch.equal(got[rank], mine)
        g = got.numpy()
        merged = np.stack([oracle.merge(g[:, i, 0], g[:, i, 1], g[:, i, 2:])[2]
                           for i in range(g.shape[1])])
        ref = oracle.attention(case.q, case.k, case.v, case.seq_lens, case.scale).reshape(
            merged.shape)
        err = float(np.max(np.abs(merged - ref)) / np.max(np.abs(ref)))
        open(os.path.join(out_dir, f"rank{rank}.txt"), "w").write(repr(err))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dcp_merge_over_gloo_ranks(world):
    # three ranks cut every sequence unevenly (301 = 100 + 100 + 101, 64 = 21 + 21 + 22)
    oracle.build()                                           # once, before the ranks start
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_dcp_rank, args=(world, _free_port(), d), nprocs=world, join=True)
        errs = [float(open(os.path.join(d, f"rank{r}.txt")).read()) for r in range(world)]
    assert max(errs) < 1e-12, errs


def _max_rank(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import importlib.util
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
        bench = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(bench)
        got = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        open(os.path.join(out_dir, f"rank{rank}.txt"), "w").write(repr(got))
    finally:
        dist.destroy_process_group()


def test_bench_time_is_the_slowest_ranks_on_gloo():
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_max_rank, args=(2, _free_port(), d), nprocs=2, join=True)
        got = [float(open(os.path.join(d, f"rank{r}.txt")).read()) for r in range(2)]
    assert got == [15.0, 15.0]


def test_context_slices_hold_the_new_tokens():
    # with q_len new tokens every slice must hold at least q_len positions
    sl = dcp.context_slices([100, 12], 3, min_len=4)
    assert all(n >= 4 for _, lens in sl for n in lens)
    with pytest.raises(ValueError):
        dcp.context_slices([100, 11], 3, min_len=4)
