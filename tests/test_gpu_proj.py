"""GPU parity of the combine fused with a per-head output projection (the MLA
value up-projection wv_b applied to the merged latent; "Attention at 128k",
§2: the output projection is a function of the merged result, so it moves into
the combine), through decode_attn_splitk_proj / decode_attn_combine_proj,
against oracle.attention_proj.

Tolerance: the attention bar (per kernel and cache type) carried through the
projection: an error of at most eps * max|V| in every merged column moves
output e by at most eps * max|V| * sum_c |W[h][e][c]|, so the bar on
|gpu - oracle| is eps * max|V| * max_{h,e} sum_c |W[h][e][c]| (plus the f32
rounding of the 128-term sums, far below it)."""
import math

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import api as A
from split_kv_decode_gb300 import workloads as W
from tests.gpu_util import TOL, to_device, vmax_per_batch

pytestmark = pytest.mark.gpu

_TDT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
MLA_BAR = {"long": 2e-4, "short": 2e-4}   # f32 latent cache: the f32 bar at every length


def proj_weights(heads, out_dim, v_dim, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((heads, out_dim, v_dim), generator=g) / math.sqrt(v_dim)).to(dtype)


def mla_case(lens, heads=96, seed=2000):
    return W.make_case("mla", batch=len(lens), n_heads=heads, n_kv_heads=1, head_dim=576,
                       v_dim=512, seq_lens=lens, kv_dtype="f32", scale=1 / math.sqrt(576.0),
                       seed=seed, std=0.5, shared_kv=True)


def bar(case, w, eps):
    row_l1 = float(w.to(torch.float64).abs().sum(dim=2).max())
    return eps * max(vmax_per_batch(case)) * row_l1


def run_proj(case, w, *, q=None, out_dtype="f32", force_splits=0, poison=True):
    qd, k, v = to_device(case)
    if q is not None:
        qd = q.cuda()
    wd = w.cuda()
    a = A.make_args(qd, k, v, case.scale, v_dim=case.v_dim, out_dtype=_TDT[out_dtype],
                    force_splits=force_splits)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    if poison:
        ws.fill_(0xFF)
    shape = tuple(qd.shape[:-1]) + (w.shape[1],)
    out = torch.full(shape, float("nan"), dtype=_TDT[out_dtype], device="cuda")
    A.decode_attn_splitk_proj(a, p, A.make_proj(wd), qd, k, v, out, ws)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    return got, (a, p, ws, qd, k, v, wd)


def worst_err(got, ref):
    return float(np.max(np.abs(got - ref)))


@pytest.mark.parametrize("wdt", [torch.float32, torch.bfloat16])
def test_mla_96_heads_wv_b_L4096(wdt):
    # 96 heads, latent 512 -> value heads of 128, f32 latent cache
    case = mla_case([4096], seed=2101)
    w = proj_weights(96, 128, 512, 2102, wdt)
    got, (a, p, *_) = run_proj(case, w)
    assert p.kernel == N.DA_KERNEL_MLA_TC
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w,
                                v_dim=512, threads=0)
    assert worst_err(got, ref) <= bar(case, w, MLA_BAR["long"])


def test_mla_96_heads_wv_b_full_context_sampled():
    case = W.named("mla_96")
    w = proj_weights(96, 128, 512, 2103)
    got, _ = run_proj(case, w)
    pairs = [(0, 0), (0, 31), (0, 47), (0, 48), (0, 95)]
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w,
                                v_dim=512, pairs=pairs, threads=0)
    g = np.stack([got[b, h] for b, h in pairs])
    assert worst_err(g, ref) <= bar(case, w, MLA_BAR["long"])


@pytest.mark.parametrize("lens", [[1, 77, 3000], [129]])
def test_mla_wv_b_short_and_ragged_contexts(lens):
    case = mla_case(lens, heads=32, seed=2104 + len(lens))
    w = proj_weights(32, 64, 512, 2105)
    got, _ = run_proj(case, w, out_dtype="f32")
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w,
                                v_dim=512, threads=0)
    assert worst_err(got, ref) <= bar(case, w, MLA_BAR["short"])


@pytest.mark.parametrize("hq,hkv,d,dtype,out_dim,wdt,out_dtype", [
    (16, 4, 256, "f16", 64, torch.bfloat16, "bf16"),
    (8, 2, 256, "f32", 256, torch.float32, "f32"),
    (32, 8, 128, "bf16", 40, torch.float32, "f16"),
    (4, 4, 128, "f16", 1, torch.bfloat16, "f32"),
])
def test_gqa_projection(hq, hkv, d, dtype, out_dim, wdt, out_dtype):
    case = W.make_case("t", batch=3, n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=[5, 1000, 7777], kv_dtype=dtype, seed=2110 + hq)
    w = proj_weights(hq, out_dim, d, 2111, wdt)
    got, _ = run_proj(case, w, out_dtype=out_dtype)
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w, threads=0)
    # plus the rounding of the output to its storage type (half an ulp, relative)
    round_rel = {"f32": 0.0, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}[out_dtype]
    assert worst_err(got, ref) <= bar(case, w, TOL[dtype]) + round_rel * float(np.max(np.abs(ref)))


@pytest.mark.parametrize("force", [1, 7, 40])
def test_projection_with_forced_splits(force):
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[3000, 9001], kv_dtype="f16", scale=1 / 16, seed=2120)
    w = proj_weights(16, 128, 256, 2121)
    got, _ = run_proj(case, w, force_splits=force)
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w, threads=0)
    assert worst_err(got, ref) <= bar(case, w, TOL["f16"])


def test_projection_with_several_new_tokens():
    case = W.make_case("t", batch=2, n_heads=8, n_kv_heads=4, head_dim=256,
                       seq_lens=[50, 4000], kv_dtype="bf16", seed=2130)
    q4 = W.multi_token_q(2, 4, 8, 256, seed=2131)
    w = proj_weights(8, 96, 256, 2132, torch.bfloat16)
    got, _ = run_proj(case, w, q=q4)
    assert got.shape == (2, 4, 8, 96)
    ref = oracle.attention_proj(q4, case.k, case.v, case.seq_lens, case.scale, w, threads=0)
    assert worst_err(got, ref) <= bar(case, w, TOL["bf16"])


def test_projection_is_the_plain_combine_followed_by_the_matrix():
    # the fused kernel and (combine, then the same per-head product on the
    # device in f64) agree to f32 rounding, and repeated runs are identical
    case = W.make_case("t", batch=1, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[20000], kv_dtype="f16", scale=1 / 16, seed=2140)
    w = proj_weights(16, 128, 256, 2141)
    got, (a, p, ws, q, k, v, wd) = run_proj(case, w)
    again, _ = run_proj(case, w)
    assert np.array_equal(got, again)
    plain = torch.empty(1, 16, 256, device="cuda")
    A.decode_attn_combine(a, p, ws, plain)
    torch.cuda.synchronize()
    want = torch.einsum("bhc,hec->bhe", plain.double(), wd.double()).cpu().numpy()
    assert worst_err(got, want) <= 1e-5 * float(np.max(np.abs(want)))


def test_projection_timed_out_weight_load_is_reported():
    # the test hook issues no weight copy: the bounded wait runs out after ~2 ms,
    # the status word names the combine and the context stays usable
    case = W.make_case("t", batch=1, n_heads=8, n_kv_heads=2, head_dim=256, seq_lens=[700],
                       kv_dtype="f32", scale=1 / 16, seed=2150)
    w = proj_weights(8, 32, 256, 2151)
    q, k, v = to_device(case)
    wd = w.cuda()
    a = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_NO_COMBINE, timeout_us=2000)
    p = A.decode_attn_plan(a, [700])
    ws = A.new_workspace(p)
    A.decode_attn_splitk_ex(a, p, q, k, v, torch.empty(1, 8, 256, device="cuda"), ws)
    a.flags = N.DA_FLAG_TEST_NO_TMA
    out = torch.empty(1, 8, 32, device="cuda")
    A.decode_attn_combine_proj(a, p, A.make_proj(wd), ws, out)
    with pytest.raises(A.DecodeAttnError) as e:
        A.decode_attn_device_status(ws)
    assert e.value.status == N.DA_ETIMEOUT
    assert "projection" in e.value.message
    got, _ = run_proj(case, w)               # the context is still usable
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w)
    assert worst_err(got, ref) <= bar(case, w, TOL["f32"])


def test_projection_over_two_context_ranks():
    # the merge of two ranks' partials (each ran the same plan on half of the
    # context) followed by the projection, against the oracle on the whole context
    from split_kv_decode_gb300 import dcp
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[6000, 2501], kv_dtype="f16", scale=1 / 16, seed=2160)
    w = proj_weights(16, 64, 256, 2161)
    lens = case.seq_lens.tolist()
    q = case.q.cuda()
    wss, plan, args = [], None, None
    for r in range(2):
        kl = dcp.shard_cache(case.k, lens, r, 2).cuda()
        vl = dcp.shard_cache(case.v, lens, r, 2).cuda()
        step = dcp.ContextParallelDecode(q, kl, vl, lens, case.scale, rank=r, world=2)
        out = torch.empty(2, 16, 256, device="cuda")
        A.decode_attn_splitk_dev(step.args, step.plan, step.dev, q, kl, vl, out, step.workspace)
        wss.append(step.workspace)
        plan, args = step.plan, step.args
    gathered = torch.stack(wss)
    out = torch.empty(2, 16, 64, device="cuda")
    A.decode_attn_combine_proj(args, plan, A.make_proj(w.cuda()), gathered, out, n_ranks=2)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    ref = oracle.attention_proj(case.q, case.k, case.v, case.seq_lens, case.scale, w, threads=0)
    assert worst_err(got, ref) <= bar(case, w, TOL["f16"])


def test_projection_in_a_captured_graph():
    # split (lengths on the device) + combine with the projection, captured once
    # and replayed over growing contexts
    case = W.make_case("t", batch=2, n_heads=16, n_kv_heads=4, head_dim=256,
                       seq_lens=[5000, 3000], kv_dtype="bf16", scale=1 / 16, seed=2170)
    w = proj_weights(16, 64, 256, 2171)
    q, k, v = to_device(case)
    wd = w.cuda()
    a = A.make_args(q, k, v, case.scale, flags=N.DA_FLAG_NO_COMBINE)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = A.new_workspace(p)
    dev_lens = torch.tensor([10, 10], dtype=torch.int32, device="cuda")
    d = A.make_dev(seq_lens=dev_lens)
    pj = A.make_proj(wd)
    out = torch.empty(2, 16, 64, device="cuda")
    scratch = torch.empty(2, 16, 256, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        A.decode_attn_splitk_dev(a, p, d, q, k, v, scratch, ws, s)
        A.decode_attn_combine_proj(a, p, pj, ws, out, stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            A.decode_attn_splitk_dev(a, p, d, q, k, v, scratch, ws, s)
            A.decode_attn_combine_proj(a, p, pj, ws, out, stream=s)
    import dataclasses
    for lens in ([10, 10], [4000, 2999], [5000, 3000]):
        dev_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        c2 = dataclasses.replace(case, seq_lens=torch.tensor(lens, dtype=torch.int32))
        ref = oracle.attention_proj(c2.q, c2.k, c2.v, c2.seq_lens, c2.scale, w, threads=0)
        assert worst_err(out.double().cpu().numpy(), ref) <= bar(c2, w, TOL["bf16"]), lens
