"""Seeded random shapes against the oracle: for each seed a random geometry
(heads per KV head, head_dim, storage type, batch, lengths from 1 to a few
thousand, new tokens per sequence, output type, forced split count) runs through
whichever kernel the plan picks, with the default two launches and with the
merge in the split kernel (DA_FLAG_ONE_LAUNCH), and every row is compared with
the oracle."""

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL

pytestmark = pytest.mark.gpu

_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
_ROUND = {"f32": 0.0, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def draw(seed):
    g = np.random.default_rng(seed)
    dtype = ["f32", "f16", "bf16"][g.integers(3)]
    d = [128, 256][g.integers(2)]
    hkv = int(g.integers(1, 5))
    gh = int(g.integers(1, 9))
    q_len = int(g.choice([1, 1, 1, 2, 3, 4]))
    # (an f32 cache with more than 8 rows per KV head runs on the SIMT kernel in
    # row groups; 16-bit caches with 8 or more on the tensor-core kernel)
    batch = int(g.integers(1, 7))
    lens = [int(x) for x in g.integers(q_len, 6000, size=batch)]
    if g.random() < 0.3:
        lens[0] = q_len                      # a sequence no longer than its new tokens
    out_dtype = ["f32", "f16", "bf16"][g.integers(3)]
    force = int(g.choice([0, 0, 0, 1, 3, 17]))
    return dtype, d, hkv, gh, q_len, batch, lens, out_dtype, force


@pytest.mark.parametrize("one_launch", [False, True])
@pytest.mark.parametrize("seed", range(24))
def test_random_shape(seed, one_launch):
    dtype, d, hkv, gh, q_len, batch, lens, out_dtype, force = draw(1000 + seed)
    hq = hkv * gh
    case = W.make_case("r", batch=batch, n_heads=hq, n_kv_heads=hkv, head_dim=d, seq_lens=lens,
                       kv_dtype=dtype, seed=2000 + seed)
    q4 = W.multi_token_q(batch, q_len, hq, d, seed=3000 + seed)
    q = q4.cuda() if q_len > 1 else q4[:, 0].contiguous().cuda()
    k, v = case.k.cuda(), case.v.cuda()
    da = A.DecodeAttention(q, k, v, lens, case.scale, out_dtype=_TDT[out_dtype],
                           force_splits=force, flags=N.DA_FLAG_ONE_LAUNCH if one_launch else 0)
    da.workspace.fill_(0xFF)
    out = da(q, k, v)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    got = out.double().cpu().numpy().reshape(batch, q_len, hq, d)
    assert np.all(np.isfinite(got))
    ref = oracle.attention_multi(q4, case.k, case.v, case.seq_lens, case.scale, threads=0)
    worst = 0.0
    for b, L in enumerate(lens):
        for t in range(q_len):
            vm = float(case.v[b, :L - q_len + 1 + t].float().abs().max())
            err = float(np.max(np.abs(got[b, t] - ref[b, t])))
            bound = TOL[dtype] * vm + _ROUND[out_dtype] * float(np.max(np.abs(ref[b, t])))
            worst = max(worst, err / bound)
    kernel = {N.DA_KERNEL_GQA_TMA: "simt", N.DA_KERNEL_GQA_TC: "tc"}[da.plan.kernel]
    assert worst <= 1.0, (dtype, d, hkv, gh, q_len, lens, out_dtype, force, kernel, one_launch,
                          worst)


@pytest.mark.parametrize("seed", range(16))
def test_random_paged_shape(seed):
    # the same random geometries over a paged pool (random block size and block
    # order, NaN in every unused block), attending over device lengths up to the
    # plan's: tiles run across block ends whatever the block size
    from tests.test_gpu_paged import paged
    dtype, d, hkv, gh, q_len, batch, lens, out_dtype, force = draw(5000 + seed)
    g = np.random.default_rng(6000 + seed)
    block_size = int(g.choice([16, 32, 48, 64, 80, 128, 256]))
    now = [int(g.integers(q_len, L + 1)) for L in lens]
    hq = hkv * gh
    case = W.make_case("p", batch=batch, n_heads=hq, n_kv_heads=hkv, head_dim=d, seq_lens=lens,
                       kv_dtype=dtype, seed=7000 + seed)
    q4 = W.multi_token_q(batch, q_len, hq, d, seed=8000 + seed)
    q = q4.cuda() if q_len > 1 else q4[:, 0].contiguous().cuda()
    kp, vp, table = paged(case, block_size, seed=seed)
    k, v, tab = kp.cuda(), vp.cuda(), table.cuda()
    a = A.make_paged_args(q, k, v, case.scale, tab.shape[1], out_dtype=_TDT[out_dtype],
                          force_splits=force)
    dev_lens = torch.tensor(now, dtype=torch.int32, device="cuda")
    dv = A.make_dev(seq_lens=dev_lens, block_table=tab, k_pool=k, v_pool=v)
    p = A.decode_attn_plan(a, lens)
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.empty(tuple(q.shape[:-1]) + (d,), dtype=_TDT[out_dtype], device="cuda")
    A.decode_attn_splitk_dev(a, p, dv, q, k, v, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    got = out.double().cpu().numpy().reshape(batch, q_len, hq, d)
    assert np.all(np.isfinite(got))
    ref = oracle.attention_multi(q4, case.k, case.v, torch.tensor(now, dtype=torch.int32),
                                 case.scale, threads=0)
    worst = 0.0
    for b, L in enumerate(now):
        for t in range(q_len):
            vm = float(case.v[b, :L - q_len + 1 + t].float().abs().max())
            err = float(np.max(np.abs(got[b, t] - ref[b, t])))
            bound = TOL[dtype] * vm + _ROUND[out_dtype] * float(np.max(np.abs(ref[b, t])))
            worst = max(worst, err / bound)
    kernel = {N.DA_KERNEL_GQA_TMA: "simt", N.DA_KERNEL_GQA_TC: "tc"}[p.kernel]
    assert worst <= 1.0, (dtype, d, hkv, gh, q_len, lens, now, block_size, out_dtype, force,
                          kernel, worst)
