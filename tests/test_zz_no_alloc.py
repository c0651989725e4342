"""The entry point that allocates nothing, decode_attn_splitk_noalloc.

It exists for callers that cannot call cudaMalloc (code that must not let
the device synchronise, hosts whose memory manager owns all device memory,
plugins without an allocator handle): the partials go to a fixed 16 MiB array
inside the library instead of a caller workspace. These checks call it
through the C ABI and compare it with decode_attn_splitk_ex, which takes a
workspace. This file is collected last on purpose.
"""
import math

import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, to_device

pytestmark = pytest.mark.gpu


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[9000, 1234], kv_dtype="f16", scale=1 / 16, seed=71)
    q, k, v = to_device(case)
    da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale)
    assert da.plan.workspace_bytes <= 16 << 20
    ref = da(q, k, v)
    torch.cuda.synchronize()
    vmax = float(case.v.float().nan_to_num(0).abs().max())
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        A.decode_attn_splitk_noalloc(da.args, da.plan, q, k, v, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        err = float((out - ref).abs().max()) / vmax
        assert err <= TOL[case.kv_dtype], err


def test_noalloc_with_another_shape_in_between():
    # the shared array keeps the previous call's contents; a call of another
    # shape in between must not leak into the next one
    small = W.make_case("t", batch=1, n_heads=8, n_kv_heads=2, head_dim=128, seq_lens=[500],
                        kv_dtype="bf16", scale=1 / math.sqrt(128), seed=73)
    big = W.make_case("t", batch=1, n_heads=24, n_kv_heads=4, head_dim=256, seq_lens=[20000],
                      kv_dtype="f32", scale=1 / 16, seed=75)
    outs = {}
    for name, case in (("big", big), ("small", small), ("big2", big)):
        q, k, v = to_device(case)
        da = A.DecodeAttention(q, k, v, case.seq_lens.tolist(), case.scale)
        ref = da(q, k, v)
        out = torch.empty_like(ref)
        A.decode_attn_splitk_noalloc(da.args, da.plan, q, k, v, out)
        torch.cuda.synchronize()
        vmax = float(case.v.float().abs().max())
        assert float((out - ref).abs().max()) / vmax <= TOL[case.kv_dtype]
        outs[name] = out.cpu()
    assert torch.equal(outs["big"], outs["big2"])


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
