"""GPU parity at the boundary's limits: the largest batch a plan holds
(DA_MAX_BATCH sequences, ragged, down to one position), the largest q_len (64
new tokens, 128 rows on the tensor-core kernel, every sequence exactly as long
as its new tokens), and the MLA kernel on a full batch."""
import math

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, run, to_device

pytestmark = pytest.mark.gpu


def _ragged(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    lens[0], lens[-1] = 1, hi
    return lens


@pytest.mark.parametrize("hq,hkv,d,dtype,kernel", [
    (8, 2, 128, "f16", N.DA_KERNEL_GQA_TMA),
    (16, 1, 128, "bf16", N.DA_KERNEL_GQA_TC),
])
def test_full_batch_of_ragged_sequences(hq, hkv, d, dtype, kernel):
    lens = _ragged(256, 1, 300, seed=1500 + hq)
    case = W.make_case("t", batch=256, n_heads=hq, n_kv_heads=hkv, head_dim=d, seq_lens=lens,
                       kv_dtype=dtype, seed=1501 + hq)
    got, da = run(case, poison_ws=True)
    assert da.plan.batch == 256 and da.plan.kernel == kernel
    assert np.all(np.isfinite(got))
    worst, rel = errors(case, got, oracle_rows(case, threads=0))
    assert worst <= TOL[dtype], (worst, rel)


def test_mla_full_batch():
    lens = _ragged(256, 1, 200, seed=1510)
    case = W.make_case("mla", batch=256, n_heads=32, n_kv_heads=1, head_dim=576, v_dim=512,
                       seq_lens=lens, kv_dtype="f32", scale=1 / math.sqrt(576.0), seed=1511,
                       std=0.5, shared_kv=True)
    got, da = run(case, poison_ws=True)
    assert da.plan.kernel == N.DA_KERNEL_MLA_TC
    worst, rel = errors(case, got, oracle_rows(case, threads=0))
    assert worst <= 2e-4, (worst, rel)   # short contexts: the f32 kernel


@pytest.mark.parametrize("lens", [[64, 64], [64, 1000]])
def test_largest_q_len(lens):
    # 64 new tokens of 2 heads over one KV head: 128 rows per item; with
    # L = 64 token 0 sees one position and token 63 all of them
    q_len = 64
    case = W.make_case("t", batch=len(lens), n_heads=2, n_kv_heads=1, head_dim=128,
                       seq_lens=lens, kv_dtype="f16", seed=1520 + lens[1])
    q4 = W.multi_token_q(len(lens), q_len, 2, 128, seed=1521)
    _, k, v = to_device(case)
    q = q4.cuda()
    da = A.DecodeAttention(q, k, v, lens, case.scale)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TC
    out = da(q, k, v)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    got = out.double().cpu().numpy()
    ref = oracle.attention_multi(q4, case.k, case.v, case.seq_lens, case.scale, threads=0)
    assert np.all(np.isfinite(got))
    worst = 0.0
    for b, L in enumerate(lens):
        for t in range(q_len):
            vm = float(case.v[b, :L - q_len + 1 + t].float().abs().max())
            worst = max(worst, float(np.max(np.abs(got[b, t] - ref[b, t]))) / vm)
    assert worst <= TOL["f16"], worst
    # token 0 of the first sequence sees position 0 alone: its output is that
    # value row, rounded only by the f32 accumulation
    assert np.allclose(got[0, 0], case.v[0, 0].double().numpy(), rtol=0, atol=1e-6)
