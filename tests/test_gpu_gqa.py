"""GPU parity of the split-KV path (split kernel + combine) against the oracle,
called through the C ABI. Sizes: every named workload, at oracle-sized
lengths for full-output checks and at full size on sampled (b, h) rows; the
boundary lengths of the pages' device tests; forced tiny chunks; edge cases."""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, run, sample_pairs, to_device

pytestmark = pytest.mark.gpu


def check(case, **kw):
    got, da = run(case, **kw)
    assert np.all(np.isfinite(got))
    ref = oracle_rows(case)
    worst, rel = errors(case, got, ref)
    assert worst <= TOL[case.kv_dtype], (worst, rel)
    return got, da, worst, rel


def check_sampled(case, per_batch=2, **kw):
    got, da = run(case, **kw)
    assert np.all(np.isfinite(got))
    pairs = sample_pairs(case, per_batch)
    ref = oracle_rows(case, pairs=pairs)
    worst, rel = errors(case, got, ref, pairs)
    assert worst <= TOL[case.kv_dtype], (worst, rel)
    return got, da, worst, rel


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------
def test_gqa_8x2_f32_L4096_full():
    check(W.named("gqa_8x2"))


@pytest.mark.parametrize("L", [4096, 20480])
def test_gqa_16x4_f16_rungs_full_output(L):
    check(W.named("gqa_16x4", seq_len=L))


@pytest.mark.parametrize("L", [61440, 151552, 262144])
def test_gqa_16x4_f16_long_rungs_sampled(L):
    check_sampled(W.named("gqa_16x4", seq_len=L), per_batch=4)


def test_gqa_24x4_f32_batch4_full_size_sampled():
    check_sampled(W.named("gqa_24x4"), per_batch=3)


def test_gqa_24x4_f32_batch4_reduced_full_output():
    check(W.named("gqa_24x4", scale_lens=1 / 32))


def test_ragged_32_bf16_reduced_full_output():
    case = W.named("ragged_32", scale_lens=1 / 32)
    check(case)


def test_ragged_32_bf16_full_size_sampled():
    check_sampled(W.named("ragged_32"), per_batch=1)


# ---------------------------------------------------------------------------
# boundary lengths and geometries (aprender issue 3725 §4 device tests;
# "Attention at 128k" §6: 12289 and 20000; gpuflight: odd length 33)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L", [1, 5, 33, 37, 64, 65, 4096, 4097, 8192, 12289, 20000])
def test_boundary_lengths_16x4_f16(L):
    check(W.make_case("t", batch=1, n_heads=16, n_kv_heads=4, head_dim=256, seq_lens=[L],
                      kv_dtype="f16", scale=1 / 16, seed=100 + L))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (24, 4), (4, 4), (8, 4), (8, 1)])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("L", [37, 4097])
def test_geometries_and_dtypes(hq, hkv, dtype, L):
    check(W.make_case("t", batch=2, n_heads=hq, n_kv_heads=hkv, head_dim=256,
                      seq_lens=[L, max(1, L // 3)], kv_dtype=dtype, scale=1 / 16,
                      seed=hq * 7 + hkv, capacity=L + 40))


# 128-wide rows in a 16-bit type are read two rows per warp step (16 lanes per
# row) for G <= 4; 301 and 5003 leave an odd number of rows in the last tile of
# some warps, so the two lane groups see different row counts
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 16), (16, 8), (48, 8), (16, 2), (64, 8)])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_head_dim_128(hq, hkv, dtype):
    check(W.make_case("t", batch=3, n_heads=hq, n_kv_heads=hkv, head_dim=128,
                      seq_lens=[1, 301, 5003], kv_dtype=dtype, seed=hq + hkv))


def test_forced_tiny_chunk_and_uneven_boundaries():
    case = W.make_case("t", batch=1, n_heads=16, n_kv_heads=4, head_dim=256, seq_lens=[4097],
                       kv_dtype="f16", scale=1 / 16, seed=3)
    for splits in (1, 3, 7, 4097):          # 4097 -> every split one tile
        got, da, worst, rel = check(case, force_splits=splits)
        assert da.plan.n_splits[0] >= 1


def test_small_sm_count_plans_run():
    case = W.make_case("t", batch=2, n_heads=8, n_kv_heads=2, head_dim=256,
                       seq_lens=[3000, 700], kv_dtype="f32", scale=1 / 16, seed=5)
    for sms in (1, 3, 40):
        check(case, num_sms=sms)


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------
def test_splitting_is_not_less_accurate_at_20000():
    # "Attention at 128k" §2.1: partials are pairwise summation; if the split
    # result were less accurate than the unsplit one, the combine would be wrong
    case = W.make_case("t", batch=1, n_heads=16, n_kv_heads=4, head_dim=256, seq_lens=[20000],
                       kv_dtype="f32", scale=1 / 16, seed=11)
    ref = oracle_rows(case)
    g_split, da = run(case)
    g_one, _ = run(case, force_splits=1)
    assert da.plan.n_splits[0] > 1
    _, rel_split = errors(case, g_split, ref)
    _, rel_one = errors(case, g_one, ref)
    print(f"relL2 split {rel_split:.3e} (S={da.plan.n_splits[0]}) vs unsplit {rel_one:.3e}")
    # measured on GB300: 2.3e-7 with 38 splits against 7.8e-7 unsplit
    assert rel_split <= rel_one


def test_f16_read_matches_the_same_values_widened_to_f32():
    # aprender issue 3725 §4: isolate the kernel's f16 read from storage rounding
    c16 = W.make_case("t", batch=1, n_heads=16, n_kv_heads=4, head_dim=256, seq_lens=[4097],
                      kv_dtype="f16", scale=1 / 16, seed=21)
    c32 = W.Case(**{**c16.__dict__, "k": c16.k.float(), "v": c16.v.float(), "kv_dtype": "f32"})
    g16, _ = run(c16)
    g32, _ = run(c32)
    assert np.max(np.abs(g16 - g32)) <= 1e-5 * float(c16.v.float().abs().max())


def test_poisoned_workspace_gives_finite_correct_output():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[5000, 77], kv_dtype="f16", scale=1 / 16, seed=23)
    check(case, poison_ws=True)


def test_poisoned_tail_past_length_is_masked():
    case = W.make_case("t", batch=2, n_heads=8, n_kv_heads=2, head_dim=256,
                       seq_lens=[333, 1000], kv_dtype="f32", scale=1 / 16, seed=29,
                       capacity=1100)
    assert torch.isnan(case.k[0, 333:]).all()
    check(case)


def test_head_major_strided_cache():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[900, 2000], kv_dtype="f16", scale=1 / 16, seed=31)
    q, k, v = to_device(case)
    kh = k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    vh = v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    got, _ = run(case, dev=(q, kh, vh))
    worst, _ = errors(case, got, oracle_rows(case))
    assert worst <= TOL["f16"]


def test_permuting_heads_within_groups_permutes_outputs():
    case = W.make_case("t", batch=1, n_heads=8, n_kv_heads=2, head_dim=256, seq_lens=[777],
                       kv_dtype="f32", scale=1 / 16, seed=37)
    base, _ = run(case)
    perm = [3, 1, 0, 2, 6, 7, 5, 4]
    c2 = W.Case(**{**case.__dict__, "q": case.q[:, perm].contiguous()})
    got, _ = run(c2)
    # a head's slot in its group sets its reduction order, so only rounding may differ
    vmax = float(case.v.float().abs().max())
    assert np.max(np.abs(got - base[:, perm])) <= 1e-6 * vmax


def test_runs_are_deterministic():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[7000, 300], kv_dtype="bf16", scale=1 / 16, seed=41)
    a, _ = run(case)
    b, _ = run(case)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("out_dtype", ["f16", "bf16"])
def test_reduced_precision_output(out_dtype):
    case = W.make_case("t", batch=2, n_heads=32, n_kv_heads=8, head_dim=128,
                       seq_lens=[5000, 1200], kv_dtype="bf16", out_dtype=out_dtype,
                       scale=1 / math.sqrt(128), seed=43)
    check(case)


# ---------------------------------------------------------------------------
# the C ABI's other entry points
# ---------------------------------------------------------------------------
def test_short_form_matches_oracle():
    case = W.make_case("t", batch=1, n_heads=16, n_kv_heads=4, head_dim=256, seq_lens=[6000],
                       kv_dtype="f32", scale=1 / 16, seed=47)
    q, k, v = to_device(case)
    out = torch.empty(1, 16, 256, device="cuda")
    A.decode_attn_splitk(q, k[0], v[0], [6000], 16, 4, 256, case.scale, out)
    torch.cuda.synchronize()
    worst, _ = errors(case, out.double().cpu().numpy(), oracle_rows(case))
    assert worst <= TOL["f32"]


def test_split_then_combine_equals_one_call():
    case = W.make_case("t", batch=2, n_heads=24, n_kv_heads=4, head_dim=256,
                       seq_lens=[9000, 4000], kv_dtype="f32", scale=1 / 16, seed=53)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale)
    one = da(q, k, v)
    args2 = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_NO_COMBINE)
    out2 = torch.full_like(one, float("nan"))
    A.decode_attn_splitk_ex(args2, da.plan, q, k, v, out2, da.workspace)
    torch.cuda.synchronize()
    assert torch.isnan(out2).all()           # the split kernel alone writes no output
    A.decode_attn_combine(args2, da.plan, da.workspace, out2)
    torch.cuda.synchronize()
    assert torch.equal(one, out2)


def test_plan_queries_the_device_sm_count():
    case = W.named("gqa_8x2")
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale)
    assert da.plan.num_sms == torch.cuda.get_device_properties(0).multi_processor_count


def test_timed_out_wait_is_reported_and_the_context_survives():
    # the producer issues no copy: every consumer wait runs out after ~2 ms and
    # the kernel reports DA_ETIMEOUT through the status word (no trap, no hang)
    case = W.make_case("t", batch=1, n_heads=8, n_kv_heads=2, head_dim=256, seq_lens=[500],
                       kv_dtype="f32", scale=1 / 16, seed=59)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, [500], case.scale, flags=N.DA_FLAG_TEST_NO_TMA,
                           timeout_us=2000)
    da(q, k, v)
    with pytest.raises(A.DecodeAttnError) as e:
        A.decode_attn_device_status(da.workspace)
    assert e.value.status == N.DA_ETIMEOUT
    assert "split" in e.value.message
    check(case)                              # the context is still usable


@pytest.mark.parametrize("shape", ["simt", "tc", "mla"])
def test_refused_launch_is_reported_and_the_context_survives(shape):
    # the test hook launches the split kernel with an empty grid: the runtime
    # refuses it before anything runs, the call returns DA_ELAUNCH naming the
    # split phase, and the next call on the same context is correct
    if shape == "mla":
        case = W.make_case("t", batch=1, n_heads=32, n_kv_heads=1, head_dim=576, v_dim=512,
                           seq_lens=[2000], kv_dtype="f32", scale=1 / math.sqrt(576.0), seed=61,
                           std=0.5, shared_kv=True)
    elif shape == "tc":
        case = W.make_case("t", batch=1, n_heads=16, n_kv_heads=1, head_dim=128,
                           seq_lens=[2000], kv_dtype="f16", seed=62)
    else:
        case = W.make_case("t", batch=1, n_heads=8, n_kv_heads=2, head_dim=256,
                           seq_lens=[2000], kv_dtype="f32", scale=1 / 16, seed=63)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, [2000], case.scale, v_dim=case.v_dim,
                           flags=N.DA_FLAG_TEST_BAD_LAUNCH)
    with pytest.raises(A.DecodeAttnError) as e:
        da(q, k, v)
    assert e.value.status == N.DA_ELAUNCH
    assert "split" in e.value.message
    got, _ = run(case)
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL[case.kv_dtype], (worst, rel)


@pytest.mark.parametrize("hq,hkv,d", [(12, 4, 256), (40, 8, 128), (14, 2, 256), (15, 5, 128)])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_odd_groups(hq, hkv, d, dtype):
    # 3, 5 and 7 query heads per KV head, ragged lengths around tile boundaries
    case = W.make_case("t", batch=3, n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=[1, 333, 5001], kv_dtype=dtype, seed=80 + hq + d)
    got, da = run(case, poison_ws=True)
    assert da.plan.kernel == N.DA_KERNEL_GQA_TMA
    worst, rel = errors(case, got, oracle_rows(case))
    assert np.all(np.isfinite(got)) and worst <= TOL[dtype], (worst, rel)
