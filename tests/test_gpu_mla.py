"""GPU parity of the MLA-as-MQA path (split kernels + combine) against the
oracle, through the C ABI.

Tolerance. The cache is f32, so every result is held to the f32 bar, 2e-4 of
max|V|. Two kernels serve the MLA shape. Sequences shorter than
DA_MLA_EXACT_BELOW (2048) positions run on the f32 CUDA-core kernel, whose
operands are all f32. Longer ones run on the tensor-core kernel, which rounds
q, the latent rows and the probabilities to bf16 and accumulates in f32; over
that many attended positions the rounding averages out, to about 1e-5 of
max|V| at 131072 positions and below 1e-4 from 2048 up. The tensor-core
kernel alone at short contexts (DA_FLAG_MLA_TC), where one value row's bf16
rounding (up to 2^-9 of it) reaches the output, is held to the 16-bit bar,
5e-3, in the tests that name that flag.
"""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import errors, oracle_rows, run, sample_pairs, to_device

pytestmark = pytest.mark.gpu

F32_BAR = 2e-4
BF16_BAR = 5e-3


def mla_case(lens, heads=96, seed=2000, cap=None, dtype="f32"):
    return W.make_case("mla", batch=len(lens), n_heads=heads, n_kv_heads=1, head_dim=576,
                       v_dim=512, seq_lens=lens, kv_dtype=dtype, scale=1 / math.sqrt(576.0),
                       seed=seed, std=0.5, shared_kv=True, capacity=cap)


def check(case, bar, **kw):
    got, da = run(case, **kw)
    assert da.plan.kernel == N.DA_KERNEL_MLA_TC
    assert np.all(np.isfinite(got))
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= bar, (worst, rel)
    return got, da, worst, rel


def test_mla_96_heads_L131072_sampled_f32_bar():
    case = W.named("mla_96")
    got, da = run(case)
    assert da.plan.kernel == N.DA_KERNEL_MLA_TC
    pairs = sample_pairs(case, per_batch=8)
    worst, rel = errors(case, got, oracle_rows(case, pairs=pairs), pairs)
    print(f"MLA L=131072: max|err|/max|V| {worst:.2e}, relL2 {rel:.2e}")
    assert worst <= F32_BAR


@pytest.mark.parametrize("L", [4096, 20000])
def test_mla_96_heads_full_output_f32_bar(L):
    check(mla_case([L], seed=2001 + L), F32_BAR)


@pytest.mark.parametrize("L", [1, 5, 31, 32, 33, 127, 128, 129, 255, 1000, 2047])
def test_mla_short_contexts(L):
    # the f32 CUDA-core kernel: f32 arithmetic throughout, so far inside the bar
    # (a bf16 operand anywhere would show at about 1e-3 here)
    got, da, worst, rel = check(mla_case([L], seed=3000 + L), F32_BAR)
    assert worst <= 1e-5, (worst, rel)


@pytest.mark.parametrize("L", [1, 5, 33, 127, 128, 129, 255, 1000])
def test_mla_tensor_core_kernel_at_short_contexts(L):
    # the tensor-core kernel forced onto short contexts: its bf16 operands
    # give the 16-bit bar here
    check(mla_case([L], seed=3000 + L), BF16_BAR, flags=N.DA_FLAG_MLA_TC)


@pytest.mark.parametrize("L,splits", [(2048, 0), (2500, 0), (3000, 5)])
def test_mla_tensor_core_kernel_just_past_the_threshold(L, splits):
    got, da, worst, rel = check(mla_case([L], seed=3300 + L), F32_BAR, force_splits=splits)
    print(f"MLA tensor cores L={L}: max|err|/max|V| {worst:.2e}, relL2 {rel:.2e}")


@pytest.mark.parametrize("L,splits", [(20000, 0), (5000, 37), (1500, 1)])
def test_mla_f32_kernel_on_request_at_any_length(L, splits):
    check(mla_case([L], seed=3400 + L), F32_BAR, flags=N.DA_FLAG_MLA_SIMT, force_splits=splits)


@pytest.mark.parametrize("heads", [32, 64])
def test_mla_fewer_heads(heads):
    check(mla_case([3000], heads=heads, seed=4000 + heads), F32_BAR)


def test_mla_batch_of_sequences_with_poisoned_tails():
    case = mla_case([700, 5000, 129], seed=5000, cap=5100)
    assert torch.isnan(case.k[0, 700:]).all()
    check(case, F32_BAR)          # 700 and 129 on the f32 kernel, 5000 on tensor cores


def test_mla_forced_splits_smaller_than_a_tile():
    for L, seed in ((2500, 5100), (1800, 5101)):   # tensor cores, then the f32 kernel
        case = mla_case([L], seed=seed)
        for s in (1, 7, 40, 157):
            got, da, worst, rel = check(case, F32_BAR, force_splits=s)
            print(f"MLA L={L} forced {s} splits: max|err|/max|V| {worst:.2e}")


def test_mla_poisoned_workspace_and_determinism():
    case = mla_case([9000], seed=5200)
    a, _, _, _ = check(case, F32_BAR, poison_ws=True)
    b, _ = run(case)
    assert np.array_equal(a, b)


def test_mla_needs_the_values_inside_the_key_rows():
    case = mla_case([300], seed=5300)
    q, k, _ = to_device(case)
    v = k.clone()
    with pytest.raises(A.DecodeAttnError) as e:
        run(case, dev=(q, k, v))
    assert e.value.status == N.DA_EUNSUPPORTED


def test_mla_timed_out_wait_is_reported_and_the_context_survives():
    # the tensor-core kernel's waits (the f32 kernel has none to run out)
    case = mla_case([3000], seed=5400)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, [3000], case.scale, v_dim=512,
                           flags=N.DA_FLAG_TEST_NO_TMA, timeout_us=2000)
    da(q, k, v)
    with pytest.raises(A.DecodeAttnError) as e:
        A.decode_attn_device_status(da.workspace)
    assert e.value.status == N.DA_ETIMEOUT and "mla" in e.value.message
    check(case, F32_BAR)


def test_mla_f32_kernel_clears_a_stale_status_word():
    # a call served by the f32 kernel alone starts from a clear status word,
    # so an earlier call's timeout is not reported again
    case = mla_case([900], seed=5410)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, [900], case.scale, v_dim=512)
    da.workspace[:4].copy_(torch.tensor([N.DA_ETIMEOUT | (N.DA_KERNEL_MLA_TC << 8)],
                                        dtype=torch.int32).view(torch.uint8).cuda())
    out = da(q, k, v)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    worst, rel = errors(case, out.double().cpu().numpy(), oracle_rows(case))
    assert worst <= F32_BAR


# ---------------------------------------------------------------------------
# several new tokens per sequence: the rows of an item are (token, head) pairs
# ---------------------------------------------------------------------------
def _multi_errors(case, q4, got, lens=None, pairs=None):
    import oracle
    lens = case.seq_lens if lens is None else torch.tensor(lens, dtype=torch.int32)
    T = q4.shape[1]
    ref = oracle.attention_multi(q4, case.k, case.v, lens, case.scale, v_dim=512, pairs=pairs,
                                 threads=0)
    worst = 0.0
    for b in range(case.batch):
        L = int(lens[b])
        for t in range(T):
            vm = float(case.k[b, :L - T + 1 + t, 0, :512].abs().max())
            if pairs is None:
                worst = max(worst, float(np.max(np.abs(got[b, t] - ref[b, t]))) / vm)
            else:
                for i, (bb, h) in enumerate(pairs):
                    if bb == b:
                        worst = max(worst, float(np.max(np.abs(got[b, t, h] - ref[t, i]))) / vm)
    return worst


def _run_multi(case, q4, force_splits=0, dev_lens=None):
    q = q4.cuda()
    k = case.k.cuda()
    a = A.make_args(q, k, k, case.scale, v_dim=512, force_splits=force_splits)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    assert p.kernel == N.DA_KERNEL_MLA_TC
    ws = A.new_workspace(p)
    ws.fill_(0xFF)
    out = torch.empty(case.batch, q4.shape[1], q4.shape[2], 512, device="cuda")
    if dev_lens is None:
        A.decode_attn_splitk_ex(a, p, q, k, k, out, ws)
    else:
        d = A.make_dev(seq_lens=torch.tensor(dev_lens, dtype=torch.int32, device="cuda"))
        A.decode_attn_splitk_dev(a, p, d, q, k, k, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    return got


@pytest.mark.parametrize("heads,q_len,lens,force", [
    (48, 2, [2, 129, 5000], 0),     # 96 rows
    (16, 4, [4, 3000], 0),          # 64 rows
    (32, 3, [3, 900, 2500], 9),     # 96 rows; short splits inside the causal tail
    (16, 2, [2, 64, 65], 0),        # 32 rows
])
def test_mla_several_new_tokens(heads, q_len, lens, force):
    case = mla_case(lens, heads=heads, seed=3100 + heads + q_len)
    q4 = W.multi_token_q(len(lens), q_len, heads, 576, seed=3101 + q_len)
    got = _run_multi(case, q4, force_splits=force)
    assert _multi_errors(case, q4, got) <= F32_BAR


def test_mla_several_new_tokens_full_context_sampled():
    # the 131072-position latent cache, 48 heads x 2 new tokens (96 rows)
    case = W.named("mla_96")
    q4 = W.multi_token_q(1, 2, 48, 576, seed=3120)
    got = _run_multi(case, q4)
    pairs = [(0, 0), (0, 23), (0, 47)]
    assert _multi_errors(case, q4, got, pairs=pairs) <= F32_BAR


def test_mla_several_new_tokens_device_lengths():
    case = mla_case([3000, 800], heads=32, seed=3130)
    q4 = W.multi_token_q(2, 2, 32, 576, seed=3131)
    got = _run_multi(case, q4, dev_lens=[2000, 1])        # 1 is kept at q_len
    assert _multi_errors(case, q4, got, lens=[2000, 2]) <= F32_BAR


def test_mla_padded_latent_rows():
    # latent rows padded to 640 elements: the kernel follows the row stride
    case = mla_case([5000], heads=64, seed=3200)
    kp = torch.zeros(1, 5000, 1, 640)
    kp[..., :576] = case.k
    k = kp.cuda()[..., :576]
    q = case.q.cuda()
    da = A.DecodeAttention(q, k, k, [5000], case.scale, v_dim=512)
    assert da.plan.kernel == N.DA_KERNEL_MLA_TC
    out = da(q, k, k)
    torch.cuda.synchronize()
    A.decode_attn_device_status(da.workspace)
    worst, rel = errors(case, out.double().cpu().numpy(), oracle_rows(case))
    assert worst <= F32_BAR, (worst, rel)


# ---------------------------------------------------------------------------
# the other MLA shapes the pages name: 128 heads, and an f16 (or bf16) latent
# cache, whose stored values are the MMA operands (the 16-bit bar, 5e-3)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L", [4096, 20000])
def test_mla_128_heads(L):
    check(mla_case([L], heads=128, seed=6000 + L), F32_BAR)


def test_mla_128_heads_L131072_sampled():
    case = W.named("mla_128")
    got, da = run(case)
    assert da.plan.kernel == N.DA_KERNEL_MLA_TC
    pairs = sample_pairs(case, per_batch=8, seed=4)
    worst, rel = errors(case, got, oracle_rows(case, pairs=pairs), pairs)
    assert worst <= F32_BAR, (worst, rel)


def test_mla_128_heads_short_contexts_on_both_kernels():
    case = mla_case([700, 129], heads=128, seed=6100)
    check(case, F32_BAR)                                  # the f32 kernel
    check(case, BF16_BAR, flags=N.DA_FLAG_MLA_TC)         # the tensor cores


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("lens", [[4096], [1, 33, 1000], [20000, 129]])
def test_mla_16bit_latent_cache(dtype, lens):
    case = mla_case(lens, heads=96, seed=6200 + len(lens), dtype=dtype)
    check(case, BF16_BAR)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_mla_16bit_latent_cache_L131072_sampled(dtype):
    case = W.named("mla_96_f16") if dtype == "f16" else mla_case([131072], dtype="bf16",
                                                                   seed=6300)
    got, da = run(case)
    pairs = sample_pairs(case, per_batch=8, seed=5)
    worst, rel = errors(case, got, oracle_rows(case, pairs=pairs), pairs)
    print(f"MLA {dtype} latent L=131072: max|err|/max|V| {worst:.2e}, relL2 {rel:.2e}")
    assert worst <= BF16_BAR, (worst, rel)


def test_mla_16bit_latent_cache_forced_splits_and_128_heads():
    case = mla_case([3000], heads=128, seed=6400, dtype="f16")
    for s in (1, 9, 150):
        check(case, BF16_BAR, force_splits=s)


def test_mla_128_rows_as_64_heads_by_2_new_tokens():
    case = mla_case([5000, 70], heads=64, seed=6500)
    q4 = W.multi_token_q(2, 2, 64, 576, seed=6501)
    got = _run_multi(case, q4)
    assert _multi_errors(case, q4, got) <= F32_BAR
