"""The entry point that allocates nothing, decode_attn_splitk_noalloc.

It exists for callers that cannot call cudaMalloc (code that must not let
the device synchronise, hosts whose memory manager owns all device memory,
plugins without an allocator handle): the partials go to a fixed 16 MiB array
inside the library instead of a caller workspace. These checks call it
through the C ABI and hold its output to the oracle element by element, with
the same bars as every other parity test, on calls in a row that share the
array. This file is collected last on purpose.
"""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, to_device

pytestmark = pytest.mark.gpu


def _noalloc(case):
    """One decode_attn_splitk_noalloc call on the case (output pre-filled with
    NaN, so an element the call does not write shows). Returns float64 numpy."""
    q, k, v = to_device(case)
    args = A.make_args(q, k, v, case.scale, v_dim=case.v_dim)
    plan = A.decode_attn_plan(args, case.seq_lens.tolist())
    assert plan.workspace_bytes <= 16 << 20
    out = torch.full((case.batch, case.n_heads, case.v_dim), float("nan"), device="cuda")
    A.decode_attn_splitk_noalloc(args, plan, q, k, v, out)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[9000, 1234], kv_dtype="f16", scale=1 / 16, seed=71)
    ref = oracle_rows(case)
    first = None
    for _ in range(2):
        got = _noalloc(case)
        assert np.all(np.isfinite(got))
        worst, rel = errors(case, got, ref)
        assert worst <= TOL[case.kv_dtype], (worst, rel)
        if first is None:
            first = got
    # the second call reuses the array the first one left behind: same plan,
    # same in-block order, so the same bits
    assert np.array_equal(first, got)


def test_noalloc_with_another_shape_in_between():
    # the shared array keeps the previous call's contents; a call of another
    # shape in between must not leak into the next one
    small = W.make_case("t", batch=1, n_heads=8, n_kv_heads=2, head_dim=128, seq_lens=[500],
                        kv_dtype="bf16", scale=1 / math.sqrt(128), seed=73)
    big = W.make_case("t", batch=1, n_heads=24, n_kv_heads=4, head_dim=256, seq_lens=[20000],
                      kv_dtype="f32", scale=1 / 16, seed=75)
    refs = {"big": oracle_rows(big), "small": oracle_rows(small)}
    outs = {}
    for name, case in (("big", big), ("small", small), ("big2", big)):
        got = _noalloc(case)
        worst, rel = errors(case, got, refs[name.rstrip("2")])
        assert worst <= TOL[case.kv_dtype], (name, worst, rel)
        outs[name] = got
    assert np.array_equal(outs["big"], outs["big2"])


def test_noalloc_refuses_plans_beyond_its_scratch():
    # 300 forced splits x 64 heads x (256 + 2) floats is about 19.8 MB > 16 MiB
    case = W.make_case("t", batch=1, n_heads=64, n_kv_heads=8, head_dim=256, seq_lens=[8400],
                       kv_dtype="f32", scale=1 / 16, seed=77)
    q, k, v = to_device(case)
    args = A.make_args(q, k, v, case.scale, force_splits=300)
    plan = A.decode_attn_plan(args, [8400])
    assert plan.workspace_bytes > 16 << 20
    out = torch.empty(1, 64, 256, device="cuda")
    with pytest.raises(A.DecodeAttnError) as e:
        A.decode_attn_splitk_noalloc(args, plan, q, k, v, out)
    assert e.value.status == N.DA_ENOSPACE
    assert "static scratch" in e.value.message
