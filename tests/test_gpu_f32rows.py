"""GPU parity of GQA/MQA over an f32 cache with 9 to 128 rows per (sequence,
KV head): large head groups, or several new tokens per group ("Decoder Block 6:
Online Attention, the Capstone", Lesson: a tile of query rows consumes each K/V
tile once). The SIMT kernel takes them with the rows cut into row groups of up
to 8, one work item each, side by side on the same K/V slice. Every operand
stays in f32, so every case is held to the f32 bar, 2e-4 of max|V|, against the
oracle, and the one-token cases to what f32 arithmetic gives."""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, run, to_device
from tests.test_gpu_multitoken import compare, run_multi

pytestmark = pytest.mark.gpu

F32_EXACT = 1e-5   # what f32 arithmetic gives; a 16-bit operand anywhere would not meet it


def case_of(hq, hkv, d, lens, seed, cap=None, layout_seed=None):
    return W.make_case("t", batch=len(lens), n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=lens, kv_dtype="f32", scale=1 / math.sqrt(d), seed=seed,
                       capacity=cap)


@pytest.mark.parametrize("hq,hkv,d", [(32, 1, 128), (24, 2, 256), (64, 4, 128), (128, 1, 128),
                                      (12, 1, 256), (11, 1, 128), (27, 1, 256)])
def test_one_token_large_groups(hq, hkv, d):
    case = case_of(hq, hkv, d, [1, 33, 2047, 9000], seed=9100 + hq + d)
    got, da = run(case, poison_ws=True)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TMA
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL["f32"], (worst, rel)
    # f32 arithmetic throughout: far inside the bar (f32 rounding of the sums
    # and the 2^x approximation, about 1e-7)
    assert worst <= F32_EXACT, (worst, rel)


@pytest.mark.parametrize("hq,hkv,q_len,d", [(16, 4, 3, 256), (8, 2, 4, 256), (16, 1, 2, 128),
                                            (24, 4, 2, 256), (64, 2, 4, 128)])
def test_several_new_tokens(hq, hkv, q_len, d):
    case = case_of(hq, hkv, d, [q_len, 70, 3001], seed=9200 + hq + q_len)
    q4 = W.multi_token_q(case.batch, q_len, hq, d, seed=9201)
    got, da = run_multi(case, q4)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TMA
    assert compare(case, q4, got) <= TOL["f32"]


def test_forced_splits_and_poisoned_tails():
    case = case_of(24, 4, 256, [333, 4000], seed=9300, cap=4100)
    assert torch.isnan(case.k[0, 333:]).all()
    q4 = W.multi_token_q(2, 2, 24, 256, seed=9301)
    for s in (1, 7, 125):
        got, da = run_multi(case, q4, force_splits=s)
        assert compare(case, q4, got) <= TOL["f32"], s


def test_head_major_cache_and_device_lengths():
    case = case_of(32, 2, 128, [5000, 600], seed=9400)
    q, k, v = to_device(case)
    # head-major copies: [B][Hkv][cap][D] viewed as [B][cap][Hkv][D]
    kh = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vh = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    a = A.make_args(q, kh, vh, case.scale)
    p = A.decode_attn_plan(a, [5000, 600])
    assert p.kernel == N.DA_KERNEL_GQA_TMA
    ws = A.new_workspace(p)
    out = torch.empty(2, 32, 128, device="cuda")
    now = [4321, 17]
    d = A.make_dev(seq_lens=torch.tensor(now, dtype=torch.int32, device="cuda"))
    A.decode_attn_splitk_dev(a, p, d, q, kh, vh, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    ref_case = case_of(32, 2, 128, [5000, 600], seed=9400)
    ref_case.seq_lens = torch.tensor(now, dtype=torch.int32)
    worst, rel = errors(ref_case, out.double().cpu().numpy(), oracle_rows(ref_case))
    assert worst <= TOL["f32"], (worst, rel)


def test_paged_pool():
    case = case_of(16, 1, 256, [3000, 129], seed=9500)
    bs, B = 64, 2
    nb = -(-3000 // bs)
    order = torch.randperm(B * nb, generator=torch.Generator().manual_seed(9501))
    table = order.view(B, nb).to(torch.int32)
    kp = torch.full((B * nb, bs, 1, 256), float("nan"))
    vp = torch.full((B * nb, bs, 1, 256), float("nan"))
    for b in range(B):
        for i in range(nb):
            lo, hi = i * bs, min((i + 1) * bs, case.capacity)
            if lo < hi:
                kp[table[b, i], :hi - lo] = case.k[b, lo:hi]
                vp[table[b, i], :hi - lo] = case.v[b, lo:hi]
    q = case.q.cuda()
    kpd, vpd = kp.cuda(), vp.cuda()
    a = A.make_paged_args(q, kpd, vpd, case.scale, nb)
    p = A.decode_attn_plan(a, [3000, 129])
    assert p.kernel == N.DA_KERNEL_GQA_TMA
    ws = A.new_workspace(p)
    out = torch.empty(2, 16, 256, device="cuda")
    d = A.make_dev(block_table=table.cuda(), k_pool=kpd, v_pool=vpd)
    A.decode_attn_splitk_dev(a, p, d, q, kpd, vpd, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    worst, rel = errors(case, out.double().cpu().numpy(), oracle_rows(case))
    assert worst <= TOL["f32"], (worst, rel)


def test_long_context_sampled():
    # the 27B-like geometry with two new tokens: 12 rows per KV head
    case = W.named("gqa_24x4", scale_lens=0.5)
    q4 = W.multi_token_q(case.batch, 2, 24, 256, seed=9601)
    got, da = run_multi(case, q4)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TMA
    pairs = [(b, h) for b in range(case.batch) for h in (0, 11, 23)]
    assert compare(case, q4, got, pairs=pairs) <= TOL["f32"]


@pytest.mark.parametrize("hq,hkv,splits", [(24, 2, 0), (32, 1, 5), (12, 1, 1)])
def test_one_launch_counts_every_row_group(hq, hkv, splits):
    # in one launch the last of a group's (split, row group) partials merges the
    # group, so the arrival count spans the row groups too
    case = case_of(hq, hkv, 256, [4000, 9, 20000], seed=9700 + hq)
    got, da = run(case, flags=N.DA_FLAG_ONE_LAUNCH, force_splits=splits, poison_ws=True)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TMA
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= F32_EXACT, (worst, rel)
