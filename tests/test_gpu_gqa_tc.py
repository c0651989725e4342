"""GPU parity of the tensor-core GQA/MQA split kernel (work items of 8 to 128
query rows on f16/bf16 caches) against the oracle, through the C ABI: single
tokens with large groups, several new tokens per sequence, the SIMT kernel on
the same 8-row shapes, forced splits, device lengths, paged pools, graph
replay and the timeout hook.

Tolerance: the 16-bit bar, 5e-3 of max|V|. The tensor-core path rounds q
(scaled) and the probabilities to the cache type and accumulates in f32."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, run, to_device

pytestmark = pytest.mark.gpu

_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
LENS = [1, 63, 64, 65, 1000, 4097]


def case_of(hq, hkv, d, dtype, lens=LENS, seed=900):
    return W.make_case("t", batch=len(lens), n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=lens, kv_dtype=dtype, seed=seed)


def check_single(case, flags=0, force_splits=0, expect=N.DA_KERNEL_GQA_TC):
    got, da = run(case, flags=flags, force_splits=force_splits, poison_ws=True)
    assert da.plan.kernel == expect
    assert np.all(np.isfinite(got))
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL[case.kv_dtype], (worst, rel)
    return got, worst


@pytest.mark.parametrize("hq,hkv,d,dtype", [
    (8, 1, 256, "f16"),      # MQA, 8 heads
    (16, 1, 128, "bf16"),    # 16 rows
    (32, 1, 128, "f16"),     # 32 rows
    (64, 1, 256, "bf16"),    # 64 rows
    (128, 1, 128, "f16"),    # 128 rows: a full M block
    (32, 4, 256, "f16"),     # 8 heads per KV head, 4 KV heads
    (64, 8, 128, "bf16"),    # 8 heads per KV head, 8 KV heads
])
def test_tensor_core_single_token(hq, hkv, d, dtype):
    check_single(case_of(hq, hkv, d, dtype, seed=900 + hq + d))


def _multi_check(case, q4, got):
    worst = 0.0
    T = q4.shape[1]
    ref = oracle.attention_multi(q4, case.k, case.v, case.seq_lens, case.scale, threads=0)
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for t in range(T):
            vm = float(case.v[b, :L - T + 1 + t].float().abs().max())
            worst = max(worst, float(np.max(np.abs(got[b, t] - ref[b, t]))) / vm)
    return worst


@pytest.mark.parametrize("hq,hkv,q_len,d,dtype", [
    (16, 4, 4, 256, "f16"),   # 16 rows
    (16, 4, 8, 256, "bf16"),  # 32 rows
    (8, 1, 16, 128, "f16"),   # 128 rows
    (4, 2, 6, 128, "bf16"),   # 12 rows (padded to 16)
])
def test_tensor_core_several_new_tokens(hq, hkv, q_len, d, dtype):
    lens = [q_len, 70, 1500, 5000]
    case = case_of(hq, hkv, d, dtype, lens=lens, seed=950 + q_len)
    q4 = W.multi_token_q(len(lens), q_len, hq, d, seed=951 + q_len)
    _, k, v = to_device(case)
    q = q4.cuda()
    da = A.DecodeAttention(q, k, v, lens, case.scale)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TC
    da.workspace.fill_(0xFF)
    out = da(q, k, v)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert _multi_check(case, q4, got) <= TOL[dtype]


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 1, 256, "f16"), (32, 4, 128, "bf16")])
def test_eight_rows_on_both_kernels(hq, hkv, d, dtype):
    case = case_of(hq, hkv, d, dtype, seed=960 + d)
    tc, e_tc = check_single(case)
    simt, e_simt = check_single(case, flags=N.DA_FLAG_GQA_SIMT, expect=N.DA_KERNEL_GQA_TMA)
    vmax = max(float(case.v.float().nan_to_num().abs().max()), 1e-30)
    assert float(np.max(np.abs(tc - simt))) / vmax <= 2 * TOL[dtype]


@pytest.mark.parametrize("force", [1, 7, 64])
def test_tensor_core_forced_splits(force):
    check_single(case_of(16, 1, 256, "f16", lens=[300, 5000], seed=970 + force),
                 force_splits=force)


def test_tensor_core_is_bit_reproducible():
    case = case_of(32, 2, 128, "bf16", lens=[9000, 3], seed=975)
    a, _ = run(case)
    b, _ = run(case)
    assert np.array_equal(a, b)


def test_tensor_core_long_context_sampled():
    # 8 query heads over one KV head, f16, 151552 positions
    case = W.make_case("t", batch=1, n_heads=8, n_kv_heads=1, head_dim=256, seq_lens=[151552],
                       kv_dtype="f16", scale=1 / 16, seed=976)
    got, da = run(case)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TC
    pairs = [(0, 0), (0, 3), (0, 7)]
    worst, rel = errors(case, got, oracle_rows(case, pairs=pairs), pairs)
    assert worst <= TOL["f16"], (worst, rel)


def _paged(case, block_size, seed=0):
    B, cap, hkv, d = case.k.shape
    nb = -(-cap // block_size)
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(B * nb + 2, generator=g)
    kp = torch.full((B * nb + 2, block_size, hkv, d), float("nan"), dtype=case.k.dtype)
    vp = torch.full_like(kp, float("nan"))
    table = torch.zeros((B, nb), dtype=torch.int32)
    for b in range(B):
        for j in range(nb):
            blk = int(order[b * nb + j])
            n = min(block_size, cap - j * block_size)
            kp[blk, :n] = case.k[b, j * block_size:j * block_size + n]
            vp[blk, :n] = case.v[b, j * block_size:j * block_size + n]
            table[b, j] = blk
    return kp, vp, table


@pytest.mark.parametrize("block_size", [16, 64, 256])
def test_tensor_core_paged_with_device_lengths(block_size):
    case = case_of(16, 2, 128, "f16", lens=[3000, 700, 1500], seed=980 + block_size)
    kp, vp, table = _paged(case, block_size, seed=block_size)
    q = case.q.cuda()
    k, v, tab = kp.cuda(), vp.cuda(), table.cuda()
    a = A.make_paged_args(q, k, v, case.scale, table.shape[1])
    lens_now = [2222, 1, 1500]
    dev_lens = torch.tensor(lens_now, dtype=torch.int32, device="cuda")
    d = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=v)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    assert p.kernel == N.DA_KERNEL_GQA_TC
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.empty(3, 16, 128, device="cuda")
    A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    got = out.double().cpu().numpy()
    ref_case = dataclasses.replace(case, seq_lens=torch.tensor(lens_now, dtype=torch.int32))
    worst, rel = errors(ref_case, got, oracle_rows(ref_case))
    assert np.all(np.isfinite(got)) and worst <= TOL["f16"], (worst, rel)


def test_tensor_core_graph_replay_over_growing_lengths():
    case = case_of(32, 1, 128, "bf16", lens=[4000, 2000], seed=990)
    q, k, v = to_device(case)
    a = A.make_args(q, k, v, case.scale)
    dev_lens = torch.tensor([100, 50], dtype=torch.int32, device="cuda")
    d = A.make_dev(seq_lens=dev_lens)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    out = torch.empty(2, 32, 128, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, s)
    for lens in ([100, 50], [1000, 1999], [4000, 2000], [1, 1]):
        dev_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        ref_case = dataclasses.replace(case, seq_lens=torch.tensor(lens, dtype=torch.int32))
        worst, rel = errors(ref_case, out.double().cpu().numpy(), oracle_rows(ref_case))
        assert worst <= TOL["bf16"], (lens, worst, rel)


def test_tensor_core_timed_out_wait_is_reported_and_the_context_survives():
    case = case_of(16, 1, 128, "f16", lens=[500], seed=995)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, [500], case.scale, flags=N.DA_FLAG_TEST_NO_TMA,
                           timeout_us=2000)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TC
    da(q, k, v)
    with pytest.raises(A.DecodeAttnError) as e:
        A.decode_attn_device_status(da.workspace)
    assert e.value.status == N.DA_ETIMEOUT
    assert "tensor cores" in e.value.message
    check_single(case)


def test_tensor_core_head_major_and_padded_caches():
    # the same values in a head-major cache, and in a position-major cache whose
    # rows are padded (strides are free as long as they are 16-byte multiples)
    case = case_of(32, 2, 128, "bf16", lens=[1000, 3001], seed=996)
    q, k, v = to_device(case)
    kh = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vh = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    got, da = run(case, dev=(q, kh, vh))
    assert da.plan.kernel == N.DA_KERNEL_GQA_TC
    worst, _ = errors(case, got, oracle_rows(case))
    assert worst <= TOL["bf16"]
    kp = torch.zeros(k.shape[0], k.shape[1], k.shape[2], 136, dtype=k.dtype, device="cuda")
    vp = torch.zeros_like(kp)
    kp[..., :128] = k
    vp[..., :128] = v
    got2, _ = run(case, dev=(q, kp[..., :128], vp[..., :128]))
    assert np.array_equal(got, got2)
