"""GPU parity of the multi-token decode (q_len > 1): q_len new tokens per
sequence, each attending causally to the cache up to its own position, served
by the GQA split kernel as extra query rows of a group that share every staged
K/V tile ("Decoder Block 6: Online Attention, the Capstone", Lesson: a tile of
query rows consumes each K/V tile once). Every result is compared with
oracle.attention_multi, token by token."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, to_device

pytestmark = pytest.mark.gpu

_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def vmax_rows(case, q_len):
    """max |V| over the rows token t of sequence b attends to, [B, q_len]."""
    out = np.zeros((case.batch, q_len))
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for t in range(q_len):
            out[b, t] = float(case.v[b, :L - q_len + 1 + t, :, :case.v_dim].float().abs().max())
    return out


def compare(case, q4, got, lens=None, pairs=None):
    """Worst |err| / max|V| over every (b, t, h) row (or the sampled pairs)."""
    lens = case.seq_lens if lens is None else torch.tensor(lens, dtype=torch.int32)
    T = q4.shape[1]
    c = dataclasses.replace(case, seq_lens=lens)
    ref = oracle.attention_multi(q4, case.k, case.v, lens, case.scale, v_dim=case.v_dim,
                                 pairs=pairs, threads=0)
    vm = vmax_rows(c, T)
    worst = 0.0
    if pairs is None:
        for b in range(case.batch):
            for t in range(T):
                e = np.max(np.abs(got[b, t] - ref[b, t])) / vm[b, t]
                worst = max(worst, float(e))
    else:
        for t in range(T):
            for i, (b, h) in enumerate(pairs):
                e = np.max(np.abs(got[b, t, h] - ref[t, i])) / vm[b, t]
                worst = max(worst, float(e))
    return worst


def run_multi(case, q4, *, force_splits=0, out_dtype="f32"):
    _, k, v = to_device(case)
    q = q4.cuda()
    da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale, v_dim=case.v_dim,
                           out_dtype=_TDT[out_dtype], force_splits=force_splits)
    da.workspace.fill_(0xFF)              # poisoned: every used partial must be written
    out = da(q, k, v)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    assert out.numel() == case.batch * q4.shape[1] * case.n_heads * case.v_dim
    got = out.view(case.batch, q4.shape[1], case.n_heads, case.v_dim).double().cpu().numpy()
    assert np.all(np.isfinite(got))
    return got, da


@pytest.mark.parametrize("hq,hkv,q_len,d,dtype", [
    (16, 4, 2, 256, "f16"),     # the default GQA shape, two tokens (group of 8 rows)
    (8, 4, 4, 256, "f32"),      # 2 heads x 4 tokens
    (8, 2, 2, 256, "bf16"),     # 4 heads x 2 tokens
    (1, 1, 6, 256, "bf16"),     # MHA head, 6 tokens
    (2, 1, 4, 128, "f16"),      # MQA pair, 4 tokens
    (32, 8, 2, 128, "bf16"),    # head_dim 128, 4 heads x 2 tokens
    (4, 4, 8, 128, "f32"),      # 8 speculative tokens per head
])
def test_multi_token_full_output(hq, hkv, q_len, d, dtype):
    lens = [q_len, 77, 1000, 5003]
    case = W.make_case("t", batch=4, n_heads=hq, n_kv_heads=hkv, head_dim=d, seq_lens=lens,
                       kv_dtype=dtype, seed=700 + hq + q_len)
    q4 = W.multi_token_q(4, q_len, hq, d, seed=701 + q_len)
    got, _ = run_multi(case, q4)
    worst = compare(case, q4, got)
    assert worst <= TOL[dtype], worst


@pytest.mark.parametrize("force", [3, 17, 64])
def test_multi_token_forced_splits_cross_the_causal_tail(force):
    # short chunks put whole splits inside the last q_len positions, where the
    # early tokens see nothing: their partials are neutral and the combine
    # must skip them
    q_len = 8
    case = W.make_case("t", batch=2, n_heads=4, n_kv_heads=4, head_dim=128,
                       seq_lens=[300, 1031], kv_dtype="f16", seed=710)
    q4 = W.multi_token_q(2, q_len, 4, 128, seed=711)
    got, da = run_multi(case, q4, force_splits=force)
    assert da.plan.n_splits[1] > 1
    assert compare(case, q4, got) <= TOL["f16"]


@pytest.mark.parametrize("out_dtype", ["f16", "bf16"])
def test_multi_token_low_precision_outputs(out_dtype):
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[2049, 4097], kv_dtype="bf16", scale=1 / 16, seed=720)
    q4 = W.multi_token_q(2, 2, 16, 256, seed=721)
    got, _ = run_multi(case, q4, out_dtype=out_dtype)
    assert compare(case, q4, got) <= 1e-2   # output rounding to 8 (bf16) bits


def test_multi_token_default_shape_full_context_sampled():
    # 16 query heads over 4 KV heads, f16, one sequence of 151552 positions,
    # two new tokens; sampled heads against the oracle
    case = W.named("gqa_16x4")
    q4 = W.multi_token_q(1, 2, 16, 256, seed=730)
    got, _ = run_multi(case, q4)
    pairs = [(0, 0), (0, 5), (0, 10), (0, 15)]
    assert compare(case, q4, got, pairs=pairs) <= TOL["f16"]


def test_multi_token_device_lengths_and_paged_pool():
    q_len, bs = 4, 64
    case = W.make_case("t", batch=3, n_heads=8, n_kv_heads=4, head_dim=256,
                       seq_lens=[3000, 700, 1500], kv_dtype="f16", seed=740, poison_tail=False)
    q4 = W.multi_token_q(3, q_len, 8, 256, seed=741)
    B, cap, hkv, d = case.k.shape
    nb = -(-cap // bs)
    g = torch.Generator().manual_seed(742)
    order = torch.randperm(B * nb + 3, generator=g)
    kp = torch.zeros((B * nb + 3, bs, hkv, d), dtype=case.k.dtype)
    vp = torch.zeros_like(kp)
    table = torch.zeros((B, nb), dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            blk = int(order[b * nb + j])
            n = min(bs, cap - j * bs)
            kp[blk, :n] = case.k[b, j * bs:j * bs + n]
            vp[blk, :n] = case.v[b, j * bs:j * bs + n]
            table[b, j] = blk
    q = q4.cuda()
    k, v, tab = kp.cuda(), vp.cuda(), table.cuda()
    a = A.make_paged_args(q, k, v, case.scale, nb)
    lens_now = [2222, 1, 1500]                 # 1 is kept at q_len on the device
    dev_lens = torch.tensor(lens_now, dtype=torch.int32, device="cuda")
    d_ = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=v)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.empty(B, q_len, 8, 256, device="cuda")
    A.decode_attn_splitk_dev(a, p, d_, q, k, v, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert compare(case, q4, got, lens=[2222, q_len, 1500]) <= TOL["f16"]


def test_single_token_in_four_dims_matches_the_three_dim_call_bit_for_bit():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[4000, 999], kv_dtype="f16", scale=1 / 16, seed=750)
    got3, _ = run_multi(case, case.q.unsqueeze(1))
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale)
    ref = da(q, k, v)
    torch.cuda.synchronize()
    assert np.array_equal(got3[:, 0], ref.double().cpu().numpy())


@pytest.mark.parametrize("hq,hkv,q_len,dtype", [(1, 1, 3, "f32"), (5, 5, 1, "bf16"),
                                                (1, 1, 5, "f16"), (1, 1, 7, "f32")])
def test_multi_token_odd_rows_on_the_simt_kernel(hq, hkv, q_len, dtype):
    lens = [q_len, 100, 2000]
    case = W.make_case("t", batch=3, n_heads=hq, n_kv_heads=hkv, head_dim=128, seq_lens=lens,
                       kv_dtype=dtype, seed=760 + q_len)
    q4 = W.multi_token_q(3, q_len, hq, 128, seed=761 + q_len)
    got, _ = run_multi(case, q4)
    assert compare(case, q4, got) <= TOL[dtype]
