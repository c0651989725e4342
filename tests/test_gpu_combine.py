"""GPU parity of the combine kernel in both its forms against the oracle: the
partials staged in shared memory by bulk copies (the default for one rank's
partials in whole 128-column blocks) and read with plain loads
(DA_FLAG_COMBINE_LOADS). Both merge by exp(m_i - m) ("Attention at 128k: Split
Over Context", §2) and skip neutral partials (l = 0), whose acc may hold
anything: the workspace is poisoned with NaN before every run."""
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, errors, oracle_rows, run, to_device

pytestmark = pytest.mark.gpu


def gqa(hq, hkv, d, lens, dt, seed, out_dtype="f32"):
    return W.make_case("t", batch=len(lens), n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=lens, kv_dtype=dt, out_dtype=out_dtype,
                       scale=1 / math.sqrt(d), seed=seed)


CASES = {
    # name: (case, forced splits)
    "f16_d256_ragged": (lambda: gqa(16, 4, 256, [9000, 77, 4096], "f16", 8700), 0),
    "bf16_d128_out_bf16": (lambda: gqa(32, 8, 128, [5000, 333, 7], "bf16", 8701, "bf16"), 0),
    "f32_d256_out_f16": (lambda: gqa(8, 2, 256, [4096, 1500], "f32", 8702, "f16"), 0),
    # more than 128 splits: the weights are formed in a second pass over (m, l)
    "f32_157_splits": (lambda: gqa(8, 2, 256, [20000], "f32", 8703), 157),
    # more than 256 splits: always the plain loads
    "f32_400_splits": (lambda: gqa(8, 2, 256, [80000], "f32", 8704), 400),
    "mla_96": (lambda: W.make_case("mla", batch=1, n_heads=96, n_kv_heads=1, head_dim=576,
                                   v_dim=512, seq_lens=[5000], kv_dtype="f32",
                                   scale=1 / math.sqrt(576.0), seed=8705, std=0.5,
                                   shared_kv=True), 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("loads", [False, True])
def test_staged_and_plain_combine_match_the_oracle(name, loads):
    make, splits = CASES[name]
    case = make()
    got, da = run(case, force_splits=splits, poison_ws=True,
                  flags=N.DA_FLAG_COMBINE_LOADS if loads else 0)
    if splits:
        assert da.plan.max_splits > (256 if splits > 300 else 128), da.plan.max_splits
    assert np.all(np.isfinite(got))
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL[case.kv_dtype], (name, loads, worst, rel)


def test_staged_and_plain_combine_agree_closely():
    # the same partials merged in both forms: the two differ only in the order
    # of the f32 sums
    case = gqa(16, 4, 256, [20000, 3000], "f16", 8710)
    q, k, v = to_device(case)
    a = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_NO_COMBINE)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    o1 = torch.empty(2, 16, 256, device="cuda")
    A.decode_attn_splitk_ex(a, p, q, k, v, o1, ws)
    o2 = torch.empty_like(o1)
    a.flags = 0
    A.decode_attn_combine(a, p, ws, o1)
    a.flags = N.DA_FLAG_COMBINE_LOADS
    A.decode_attn_combine(a, p, ws, o2)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    scale = float(o2.abs().max())
    assert float((o1 - o2).abs().max()) <= 1e-6 * scale


def test_staged_combine_timed_out_wait_is_reported_and_the_context_survives():
    # the test hook issues no bulk copy, so the combine's bounded wait runs out
    case = gqa(8, 2, 256, [700], "f32", 8720)
    q, k, v = to_device(case)
    a = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_NO_COMBINE, timeout_us=2000)
    p = A.decode_attn_plan(a, [700])
    ws = A.new_workspace(p)
    out = torch.empty(1, 8, 256, device="cuda")
    A.decode_attn_splitk_ex(a, p, q, k, v, out, ws)
    a.flags = N.DA_FLAG_TEST_NO_TMA
    A.decode_attn_combine(a, p, ws, out)
    with pytest.raises(A.DecodeAttnError) as e:
        A.decode_attn_device_status(ws)
    assert e.value.status == N.DA_ETIMEOUT
    assert "combine" in e.value.message and "projection" not in e.value.message
    got, _ = run(case)                       # the context is still usable
    worst, rel = errors(case, got, oracle_rows(case))
    assert worst <= TOL["f32"], (worst, rel)
