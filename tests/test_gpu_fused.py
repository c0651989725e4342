"""GPU parity of the one-launch step (DA_FLAG_ONE_LAUNCH), in which the split
kernel merges its own partials (no combine launch), against the oracle.

The GQA kernels count the arrivals of each (sequence, KV head) group's
partials, and every CTA, after its own arrivals, waits for its items' groups
and merges a share of each. The MLA tensor-core kernel counts the arrivals of
all its CTAs; then every CTA stages its share of the rows in shared memory and
merges it. The library zeroes the counters on the stream before each such launch, so
a poisoned workspace, a workspace shared by calls of other shapes and a CUDA
graph replay all start from zero. Each case is checked against the oracle in
both forms (one launch, and the default two launches) with the same bars as
the other parity tests.
"""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, run, sample_pairs, to_device

pytestmark = pytest.mark.gpu


def mla_case(lens, heads=96, seed=8000):
    return W.make_case("mla", batch=len(lens), n_heads=heads, n_kv_heads=1, head_dim=576,
                       v_dim=512, seq_lens=lens, kv_dtype="f32", scale=1 / math.sqrt(576.0),
                       seed=seed, std=0.5, shared_kv=True)


CASES = {
    "simt_f16": lambda: W.make_case("t", batch=3, n_heads=16, n_kv_heads=4, head_dim=256,
                                    seq_lens=[9000, 77, 4096], kv_dtype="f16", scale=1 / 16,
                                    seed=8100),
    "simt_f32_g2": lambda: W.make_case("t", batch=2, n_heads=8, n_kv_heads=4, head_dim=256,
                                       seq_lens=[3000, 20000], kv_dtype="f32", scale=1 / 16,
                                       seed=8101),
    "simt_bf16_d128_out_bf16": lambda: W.make_case(
        "t", batch=5, n_heads=32, n_kv_heads=8, head_dim=128, seq_lens=[1024, 5000, 333, 7, 12000],
        kv_dtype="bf16", out_dtype="bf16", scale=1 / math.sqrt(128), seed=8102),
    "tc_bf16_d128": lambda: W.make_case("t", batch=2, n_heads=32, n_kv_heads=2, head_dim=128,
                                        seq_lens=[3000, 65], kv_dtype="bf16", seed=8103),
    "mla_96": lambda: mla_case([5000], seed=8104),
    "mla_64_batch": lambda: mla_case([2100, 9000, 4000], heads=64, seed=8105),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("two_launch", [False, True])
def test_one_launch_and_two_launch_match_the_oracle(name, two_launch):
    case = CASES[name]()
    got, da = run(case, flags=0 if two_launch else N.DA_FLAG_ONE_LAUNCH, poison_ws=True)
    worst, rel = errors(case, got, oracle_rows(case))
    assert np.all(np.isfinite(got))
    assert worst <= TOL[case.kv_dtype], (name, two_launch, worst, rel)


@pytest.mark.parametrize("splits", [1, 3, 157])
def test_one_launch_with_forced_splits(splits):
    case = W.make_case("t", batch=2, n_heads=24, n_kv_heads=4, head_dim=256,
                       seq_lens=[6000, 2600], kv_dtype="f32", scale=1 / 16, seed=8200)
    got, da = run(case, force_splits=splits, flags=N.DA_FLAG_ONE_LAUNCH)
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL["f32"], (splits, worst, rel)


@pytest.mark.parametrize("splits", [1, 100])
def test_one_launch_tensor_cores_with_forced_splits(splits):
    # the shares of a group merge 100 splits in two batches of 64 per lane group
    case = W.make_case("t", batch=2, n_heads=32, n_kv_heads=2, head_dim=128,
                       seq_lens=[20000, 3000], kv_dtype="bf16", seed=8210)
    got, da = run(case, force_splits=splits, flags=N.DA_FLAG_ONE_LAUNCH, poison_ws=True)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TC
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL["bf16"], (splits, worst, rel)


def test_one_launch_mla_full_context_sampled():
    case = W.named("mla_96")
    got, da = run(case, flags=N.DA_FLAG_ONE_LAUNCH)
    pairs = sample_pairs(case, per_batch=6, seed=3)
    worst, rel = errors(case, got, oracle_rows(case, pairs=pairs), pairs)
    assert worst <= TOL["f32"], (worst, rel)


@pytest.mark.parametrize("heads,splits", [(128, 0), (96, 300), (32, 0), (64, 7)])
def test_one_launch_mla_staged_passes(heads, splits):
    # each CTA stages its (row, 128 columns) units in shared memory: with 128
    # heads a CTA's units take two passes; with 300 splits one unit outgrows
    # the stage and is merged from L2 instead; the workspace is poisoned, so a
    # neutral partial's unwritten acc would show
    case = mla_case([20000], heads=heads, seed=8600 + heads + splits)
    got, da = run(case, flags=N.DA_FLAG_ONE_LAUNCH, force_splits=splits, poison_ws=True)
    worst, rel = errors(case, got, oracle_rows(case))
    assert np.all(np.isfinite(got))
    assert worst <= TOL["f32"], (heads, splits, worst, rel)


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_one_launch_replayed_from_a_cuda_graph(kind):
    # a graph replays the counter reset and the launch together, so every
    # replay merges exactly once
    if kind == "mla":
        case = mla_case([6000], heads=32, seed=8300)
    else:
        case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                           seq_lens=[7000, 3001], kv_dtype="f16", scale=1 / 16, seed=8301)
    q, k, v = to_device(case)
    a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, flags=N.DA_FLAG_ONE_LAUNCH)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.empty(case.batch, case.n_heads, case.v_dim, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        A.decode_attn_splitk_ex(a, p, q, k, v, out, ws, s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            A.decode_attn_splitk_ex(a, p, q, k, v, out, ws, s)
    torch.cuda.synchronize()
    ref = oracle_rows(case)
    for i in range(4):
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        A.decode_attn_device_status(ws)
        worst, rel = errors(case, out.double().cpu().numpy(), ref)
        assert worst <= TOL[case.kv_dtype], (i, worst, rel)


def test_one_launch_workspace_shared_by_calls_of_other_shapes():
    # the counters of one plan lie over another plan's partials: each call
    # zeroes its own before its launch
    big = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                      seq_lens=[9000, 5000], kv_dtype="f16", scale=1 / 16, seed=8400)
    small = W.make_case("t", batch=3, n_heads=8, n_kv_heads=2, head_dim=256,
                        seq_lens=[300, 4000, 12], kv_dtype="f16", scale=1 / 16, seed=8401)
    ws = None
    for case in (big, small, big, small):
        q, k, v = to_device(case)
        a = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_ONE_LAUNCH)
        p = A.decode_attn_plan(a, case.seq_lens.tolist())
        if ws is None:
            ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
        out = torch.full((case.batch, case.n_heads, case.v_dim), float("nan"), device="cuda")
        A.decode_attn_splitk_ex(a, p, q, k, v, out, ws)
        torch.cuda.synchronize()
        A.decode_attn_device_status(ws)
        worst, rel = errors(case, out.double().cpu().numpy(), oracle_rows(case))
        assert worst <= TOL["f16"], (worst, rel)


@pytest.mark.parametrize("kind", ["simt", "tc"])
def test_one_launch_plan_wider_than_the_gpu_falls_back_to_the_combine(kind):
    # a plan made for more SMs than the device has gives a grid that is not
    # resident at once: the GQA kernels then leave the merge to the combine
    # launch, and the result still matches the oracle
    hq, hkv, dt = (16, 4, "f16") if kind == "simt" else (32, 2, "f16")
    case = W.make_case("t", batch=2, n_heads=hq, n_kv_heads=hkv, head_dim=256,
                       seq_lens=[30000, 9000], kv_dtype=dt, scale=1 / 16, seed=8500)
    q, k, v = to_device(case)
    a = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_ONE_LAUNCH)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = A.decode_attn_plan(a, case.seq_lens.tolist(), num_sms=4 * sms)
    want = N.DA_KERNEL_GQA_TMA if kind == "simt" else N.DA_KERNEL_GQA_TC
    assert p.kernel == want and p.grid > sms
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.full((case.batch, case.n_heads, case.v_dim), float("nan"), device="cuda")
    A.decode_attn_splitk_ex(a, p, q, k, v, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    worst, rel = errors(case, out.double().cpu().numpy(), oracle_rows(case))
    assert worst <= TOL["f16"], (worst, rel)
