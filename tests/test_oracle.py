"""Pins for the double-precision oracle (CPU only).

Each check ties the oracle to something other than itself: closed forms,
the independent numpy brute force, the split identity the pages state, the
page's worked merge example, and negative controls that plant the pages'
named mistakes in the oracle and require the checks to catch them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from split_kv_decode_gb300 import workloads as W
from tests._naive import naive_attention, naive_causal_attention, widen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def vmax(case):
    x = widen(case.v)
    x = x[np.isfinite(x)]
    return float(np.max(np.abs(x)))


def small(hq, hkv, d, lens, dtype="f32", dv=None, seed=7, scale=None, cap=None, std=1.0,
          shared=False):
    return W.make_case("t", batch=len(lens), n_heads=hq, n_kv_heads=hkv, head_dim=d,
                       seq_lens=lens, kv_dtype=dtype, v_dim=dv, seed=seed, scale=scale,
                       capacity=cap, std=std, shared_kv=shared)


def run_oracle(c, **kw):
    return oracle.attention(c.q, c.k, c.v, c.seq_lens, c.scale, v_dim=c.v_dim, **kw)


# ---------------------------------------------------------------------------
# brute force on tiny inputs, every geometry and storage type
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (4, 2), (8, 2), (6, 1), (12, 2), (16, 4),
                                    (9, 3), (15, 3), (14, 2)])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_brute_force_agreement(hq, hkv, dtype):
    c = small(hq, hkv, 16, [1, 5, 33, 64], dtype=dtype, cap=70, scale=0.7, seed=hq * 31 + hkv)
    ref = naive_attention(c.q, c.k, c.v, c.seq_lens, c.scale)
    got = run_oracle(c)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) <= 1e-13 * vmax(c)


def test_brute_force_separate_value_width():
    c = small(6, 2, 16, [9, 40], dv=8, cap=41, seed=3)
    ref = naive_attention(c.q, c.k, c.v, c.seq_lens, c.scale)
    got = run_oracle(c)
    assert got.shape == (2, 6, 8)
    assert np.max(np.abs(got - ref)) <= 1e-13 * vmax(c)


def test_brute_force_shared_latent_mla_shape():
    # MLA as MQA: one latent row per position, values = its first v_dim columns
    c = small(6, 1, 24, [37], dv=16, seed=11, std=0.5, shared=True, scale=1 / math.sqrt(24))
    assert c.k.data_ptr() == c.v.data_ptr()
    ref = naive_attention(c.q, c.k, c.k, c.seq_lens, c.scale, v_dim=16)
    got = run_oracle(c)
    assert np.max(np.abs(got - ref)) <= 1e-13 * vmax(c)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_zero_query_gives_mean_of_values(dtype):
    c = W.make_case("t", batch=2, n_heads=4, n_kv_heads=2, head_dim=16, seq_lens=[7, 50],
                    kv_dtype=dtype, seed=5, q_zero=True, capacity=64)
    got = run_oracle(c)
    V = widen(c.v)
    for b in range(2):
        L = int(c.seq_lens[b])
        for h in range(4):
            mean = V[b, :L, h // 2, :].mean(axis=0)
            assert np.max(np.abs(got[b, h] - mean)) <= 1e-14 * vmax(c)


def test_dominant_score_selects_that_row():
    c = small(4, 1, 16, [64], std=0.01, seed=9, scale=0.25)
    jstar = 37
    q = c.q[0, 2].clone()
    c.k[0, jstar, 0] = q * (100.0 / (c.scale * float(q.dot(q))))   # s_j* = 100, others ~0
    got = run_oracle(c)
    V = widen(c.v)
    assert np.max(np.abs(got[0, 2] - V[0, jstar, 0])) <= 1e-15
    # the other heads of the group do not see it as dominant
    assert np.max(np.abs(got[0, 0] - V[0, jstar, 0])) > 1e-3


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_single_position_returns_value_row_exactly(dtype):
    c = small(8, 2, 16, [1, 1], dtype=dtype, cap=3, seed=13)
    got = run_oracle(c)
    V = widen(c.v)
    for b in range(2):
        for h in range(8):
            assert np.array_equal(got[b, h], V[b, 0, h // 4])


def test_storage_readers_on_special_values():
    # L = 1 makes out = V row 0 exactly; the row holds edge values of each format
    f16_vals = [2.0 ** -24, 2.0 ** -14, 65504.0, -0.0, -1.5, 1.0 / 3.0, 2.0 ** -20, -2.0 ** -24]
    bf16_vals = [1e-40, -3.0e38, 2.0 ** -126, 1.0 / 3.0, -7.25, 0.0, 1e30, 2.0 ** -133]
    for vals, dt in ((f16_vals, torch.float16), (bf16_vals, torch.bfloat16)):
        v = torch.tensor(vals, dtype=torch.float32).to(dt).reshape(1, 1, 1, -1)
        k = torch.zeros_like(v)
        q = torch.zeros(1, 1, v.shape[-1])
        got = oracle.attention(q, k, v, [1], 1.0)
        assert np.array_equal(got[0, 0], v.double().numpy()[0, 0, 0])


def test_permuting_heads_within_a_group_permutes_outputs():
    c = small(8, 2, 16, [45], seed=17)
    base = run_oracle(c)
    perm = [2, 0, 3, 1, 7, 5, 4, 6]          # stays inside each group of 4
    c2 = W.Case(**{**c.__dict__, "q": c.q[:, perm].contiguous()})
    got = run_oracle(c2)
    assert np.array_equal(got, base[:, perm])


def test_swapping_kv_heads_with_their_groups():
    c = small(6, 3, 16, [30], seed=19)
    base = run_oracle(c)
    qperm = [4, 5, 0, 1, 2, 3]               # groups (0,1),(2,3),(4,5) -> kv 2,0,1
    kperm = [2, 0, 1]
    c2 = W.Case(**{**c.__dict__, "q": c.q[:, qperm].contiguous(),
                   "k": c.k[:, :, kperm].contiguous(), "v": c.v[:, :, kperm].contiguous()})
    assert np.array_equal(run_oracle(c2), base[:, qperm])


def test_strided_head_major_layout_matches():
    c = small(4, 2, 16, [20, 33], cap=40, seed=23)
    base = run_oracle(c)
    kh = c.k.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)   # head-major storage
    vh = c.v.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert not kh.is_contiguous()
    got = oracle.attention(c.q, kh, vh, c.seq_lens, c.scale)
    assert np.array_equal(got, base)


def test_pairs_and_threads_do_not_change_rows():
    c = small(8, 2, 16, [20, 33, 7], cap=40, seed=29)
    base = run_oracle(c, threads=1)
    assert np.array_equal(run_oracle(c, threads=4), base)
    pairs = [(2, 7), (0, 0), (1, 3)]
    got = run_oracle(c, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(got[i], base[b, h])


def test_masking_ignores_positions_past_length():
    # positions past seq_len hold NaN; any read of them would poison the row
    c = small(4, 2, 16, [3, 17], cap=32, seed=31)
    assert torch.isnan(c.k[0, 3:]).all()
    assert np.all(np.isfinite(run_oracle(c)))


def test_invalid_arguments_are_rejected():
    c = small(4, 2, 16, [5], seed=1)
    with pytest.raises(ValueError):
        oracle.attention(c.q, c.k, c.v, [0], c.scale)
    with pytest.raises(ValueError):
        oracle.attention(c.q, c.k, c.v, [6], c.scale)


# ---------------------------------------------------------------------------
# the split identity ("exact up to floating-point reassociation")
# ---------------------------------------------------------------------------
def split_error(c, n_splits, block, form=oracle.MERGE_ML, flags=0):
    full = run_oracle(c)
    sp = oracle.attention_split(c.q, c.k, c.v, c.seq_lens, c.scale, n_splits, block=block,
                                form=form, flags=flags, v_dim=c.v_dim)
    return np.max(np.abs(sp - full)) / vmax(c)


@pytest.mark.parametrize("n_splits", [1, 2, 3, 7, 64, 97, 102])
@pytest.mark.parametrize("block", [1, 5, 32, 64])
@pytest.mark.parametrize("form", [oracle.MERGE_ML, oracle.MERGE_LSE])
def test_split_identity(n_splits, block, form):
    c = small(4, 2, 16, [97, 50], cap=100, seed=37, scale=1.0)   # scores ~ N(0, 16)
    assert split_error(c, n_splits, block, form) <= 1e-12


def test_split_identity_dtypes_and_mla_shape():
    for c in (small(12, 2, 16, [200], dtype="bf16", seed=41),
              small(8, 2, 16, [129], dtype="f16", seed=43),
              small(6, 1, 24, [150], dv=16, std=0.5, shared=True, seed=47)):
        for s in (1, 3, 16, 150):
            assert split_error(c, s, 32) <= 1e-12


def test_empty_segments_are_neutral():
    c = small(4, 2, 16, [5, 3], cap=8, seed=53)
    # 8 splits over 5 and 3 positions: trailing segments are empty
    out, pm, pl, pO = oracle.attention_split(c.q, c.k, c.v, c.seq_lens, c.scale, 8,
                                             return_partials=True)
    assert np.all(np.isfinite(out))
    b1_rows = slice(4, 8)                       # batch element 1, L = 3
    assert np.all(pl[b1_rows, 3:] == 0.0) and np.all(pm[b1_rows, 3:] == -1e30)
    assert np.all(pO[b1_rows, 3:] == 0.0)
    assert np.max(np.abs(out - run_oracle(c))) <= 1e-13 * vmax(c)


def test_partials_are_the_segment_triples():
    # m_s = max s_j, l_s = sum e^{s_j - m_s}, O_s = sum e^{s_j - m_s} v_j over each segment
    c = small(2, 1, 8, [30], seed=59, scale=1.0)
    _, pm, pl, pO = oracle.attention_split(c.q, c.k, c.v, c.seq_lens, c.scale, 3, block=4,
                                           return_partials=True)
    Q, K, V = widen(c.q), widen(c.k), widen(c.v)
    for h in range(2):
        s = (K[0, :30, 0] @ Q[0, h]) * c.scale
        for seg in range(3):
            ss, vv = s[seg * 10:(seg + 1) * 10], V[0, seg * 10:(seg + 1) * 10, 0]
            m = ss.max()
            assert abs(pm[h, seg] - m) <= 1e-14 * abs(m)
            assert abs(pl[h, seg] - np.exp(ss - m).sum()) <= 1e-13 * pl[h, seg]
            assert np.max(np.abs(pO[h, seg] - np.exp(ss - m) @ vv)) <= 1e-13 * np.abs(vv).max() * 10



@pytest.mark.parametrize("form", [oracle.MERGE_ML, oracle.MERGE_LSE])
@pytest.mark.parametrize("groups", [[4, 4, 4], [1, 11], [5, 2, 5], [3, 3, 3, 3]])
def test_merging_in_groups_equals_merging_at_once(form, groups):
    # Context-parallel decode merges each rank's splits and then the ranks
    # ("The Kernel Level": DCP is split-KV at another scale). A merged row is a
    # partial again -- (m, l, O = out * l), or (LSE*, 1, out) for the LSE form --
    # so any grouping of the 12 segments must give the one-level result.
    c = small(4, 2, 16, [120], cap=120, seed=61, scale=1.0)
    ref, pm, pl, pO = oracle.attention_split(c.q, c.k, c.v, c.seq_lens, c.scale, 12, block=8,
                                             return_partials=True)
    ref = ref.reshape(4, -1)
    for row in range(4):
        mg, lg, Og, i = [], [], [], 0
        for n in groups:
            m1, l1, out1 = oracle.merge(pm[row, i:i + n], pl[row, i:i + n], pO[row, i:i + n],
                                        form=form)
            mg.append(m1)
            lg.append(l1)
            Og.append(out1 * l1)
            i += n
        _, _, out = oracle.merge(mg, lg, np.stack(Og), form=form)
        assert np.max(np.abs(out - ref[row])) <= 1e-12 * np.abs(ref[row]).max()

# ---------------------------------------------------------------------------
# negative controls: the planted mistakes must be caught
# ---------------------------------------------------------------------------
def test_negative_control_merge_without_rescale_is_caught():
    c = small(4, 2, 16, [97, 50], cap=100, seed=37, scale=1.0)
    assert split_error(c, 7, 32) <= 1e-12
    assert split_error(c, 7, 32, flags=oracle.NC_NO_MERGE_RESCALE) > 1e-3


def test_negative_control_missing_alpha_at_length_33_is_caught():
    # two tiles of 32; the running max moves in the second tile (position 32)
    c = small(2, 1, 16, [33], seed=61, scale=0.25)
    c.k[0, 32, 0] = c.q[0, 0] * (8.0 / (c.scale * float(c.q[0, 0].dot(c.q[0, 0]))))
    assert split_error(c, 1, 32) <= 1e-12
    assert split_error(c, 1, 32, flags=oracle.NC_NO_ALPHA) > 1e-3


# ---------------------------------------------------------------------------
# the worked merge example of "The Kernel Level" page
# ---------------------------------------------------------------------------
def _worked_example():
    with open(os.path.join(GOLDEN, "merge_worked_example.json")) as f:
        return json.load(f)


def test_worked_merge_example_matches_brute_force():
    ex = _worked_example()
    m = [p["m"] for p in ex["partials"]]
    l = [p["l"] for p in ex["partials"]]
    O = [p["O"] for p in ex["partials"]]
    # a concrete score/value set with exactly these block statistics:
    # block 1: eight scores equal to 2 with values 0.5 (l = 8, O = 4);
    # block 2: six scores equal to 3 with values 3 (l = 6, O = 18)
    s = np.array([2.0] * 8 + [3.0] * 6)
    vals = np.array([0.5] * 8 + [3.0] * 6)
    assert np.exp(s[:8] - 2).sum() == l[0] and (np.exp(s[:8] - 2) * vals[:8]).sum() == O[0][0]
    assert np.exp(s[8:] - 3).sum() == l[1] and (np.exp(s[8:] - 3) * vals[8:]).sum() == O[1][0]
    q = np.ones((1, 1, 1))
    K = s.reshape(1, -1, 1, 1)
    V = vals.reshape(1, -1, 1, 1)
    want = naive_attention(q, K, V, [14], 1.0)[0, 0]
    for form in (oracle.MERGE_ML, oracle.MERGE_LSE):
        mm, ll, out = oracle.merge(m, l, O, form=form)
        assert abs(out[0] - want[0]) <= 1e-15 * abs(want[0])
    mm, ll, out = oracle.merge(m, l, O)
    assert mm == 3.0
    assert abs(ll - np.exp(s - 3.0).sum()) <= 1e-15 * ll
    # reading O_1 as already normalised would give a different answer
    mis = (8 * math.exp(-1) * 4 + 6 * 3) / (8 * math.exp(-1) + 6)
    assert abs(out[0] - mis) > 0.5


def test_worked_example_with_a_neutral_third_partial():
    ex = _worked_example()
    m = [p["m"] for p in ex["partials"]]
    l = [p["l"] for p in ex["partials"]]
    O = [p["O"] for p in ex["partials"]]
    _, _, ref = oracle.merge(m, l, O)
    for order in ((0, 1, 2), (2, 1, 0), (1, 2, 0)):
        mm = [(m + [-1e30])[i] for i in order]
        lll = [(l + [0.0])[i] for i in order]
        OO = [(O + [[0.0]])[i] for i in order]
        _, _, got = oracle.merge(mm, lll, OO)
        assert np.isfinite(got[0]) and abs(got[0] - ref[0]) <= 1e-15 * abs(ref[0])
    with pytest.raises(ValueError):
        oracle.merge([-1e30, -1e30], [0.0, 0.0], [[0.0], [0.0]])


# ---------------------------------------------------------------------------
# several new tokens per sequence, causal among themselves
# ---------------------------------------------------------------------------
def _multi(hq, hkv, d, lens, T, dtype="f32", seed=11, scale=0.6):
    c = small(hq, hkv, d, lens, dtype=dtype, cap=max(lens) + 3, seed=seed, scale=scale)
    return c, W.multi_token_q(len(lens), T, hq, d, seed=seed + 1)


@pytest.mark.parametrize("hq,hkv,T", [(1, 1, 2), (4, 2, 3), (8, 2, 4), (6, 1, 2), (16, 4, 2)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_token_brute_force_with_explicit_mask(hq, hkv, T, dtype):
    c, q = _multi(hq, hkv, 16, [T, 7, 40], T, dtype=dtype, seed=hq + 3 * T)
    ref = naive_causal_attention(q, c.k, c.v, c.seq_lens, c.scale)
    got = oracle.attention_multi(q, c.k, c.v, c.seq_lens, c.scale)
    assert got.shape == (3, T, hq, 16)
    assert np.max(np.abs(got - ref)) <= 1e-13 * vmax(c)


def test_multi_token_whole_sequence_first_token_sees_only_position_zero():
    # q_len = L: the prefill of the whole sequence; token 0 attends to position 0
    # alone, so its output is that value row exactly
    c, q = _multi(4, 2, 8, [6], 6, seed=5)
    got = oracle.attention_multi(q, c.k, c.v, c.seq_lens, c.scale)
    for h in range(4):
        assert np.array_equal(got[0, 0, h], widen(c.v[0, 0, h // 2]))
    ref = naive_causal_attention(q, c.k, c.v, c.seq_lens, c.scale)
    assert np.max(np.abs(got - ref)) <= 1e-13 * vmax(c)


def test_multi_token_last_token_is_single_token_decode():
    c, q = _multi(8, 2, 16, [9, 33], 3, seed=9)
    got = oracle.attention_multi(q, c.k, c.v, c.seq_lens, c.scale)
    one = oracle.attention(q[:, -1], c.k, c.v, c.seq_lens, c.scale)
    assert np.array_equal(got[:, -1], one)
    # and one token is the single-token call itself
    got1 = oracle.attention_multi(q[:, :1], c.k, c.v, c.seq_lens, c.scale)
    assert np.array_equal(got1[:, 0], oracle.attention(q[:, 0], c.k, c.v, c.seq_lens, c.scale))


def test_multi_token_negative_control_off_by_one_mask_is_caught():
    # a mask that lets token t see one position too many (or too few) differs
    c, q = _multi(4, 1, 16, [12], 3, seed=13)
    ref = naive_causal_attention(q, c.k, c.v, c.seq_lens, c.scale)
    for shift in (1, -1):
        bad = np.stack([oracle.attention(q[:, t], c.k, c.v,
                                         np.array([12 - 3 + 1 + t + shift], dtype=np.int32),
                                         c.scale) for t in range(2)], axis=1)
        assert np.max(np.abs(bad - ref[:, :2])) > 1e-3


def test_multi_token_rejects_short_sequences():
    c, q = _multi(2, 1, 8, [2, 9], 3, seed=2)
    with pytest.raises(ValueError):
        oracle.attention_multi(q, c.k, c.v, c.seq_lens, c.scale)


# ---------------------------------------------------------------------------
# attention followed by a per-head projection (wv_b)
# ---------------------------------------------------------------------------
def _proj_weights(h, e, c, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((h, e, c), generator=g) / math.sqrt(c)).to(dtype)


def test_projection_equals_attention_over_projected_values():
    # (P V) W^T = P (V W^T): project every value row with head h's matrix first,
    # then run materialised attention for that head alone
    c = small(6, 1, 24, [1, 9, 40], dv=16, cap=41, seed=21, shared=True)
    W_ = _proj_weights(6, 8, 16, 22)
    got = oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, W_, v_dim=16)
    Wn = widen(W_)
    V = widen(c.v)[..., :16]
    for h in range(6):
        Vh = np.einsum("bpkc,ec->bpke", V, Wn[h])            # [B, cap, 1, out]
        ref = naive_attention(widen(c.q)[:, h:h + 1], widen(c.k), Vh, c.seq_lens, c.scale)
        assert np.max(np.abs(got[:, h] - ref[:, 0])) <= 1e-13 * np.max(np.abs(ref))


def test_projection_identity_and_selectors_are_exact():
    c = small(4, 2, 16, [5, 33], seed=23)
    att = run_oracle(c)
    eye = torch.eye(16).expand(4, 16, 16).contiguous()
    assert np.array_equal(oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, eye), att)
    sel = torch.zeros(4, 3, 16)
    for h in range(4):
        for e, col in enumerate((h, 15 - h, 7)):
            sel[h, e, col] = 1.0
    got = oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, sel)
    for h in range(4):
        assert np.array_equal(got[:, h], att[:, h][:, [h, 15 - h, 7]])


def test_projection_bf16_weights_widen_exactly_and_pairs_match():
    c = small(4, 1, 16, [12, 30], seed=25)
    Wb = _proj_weights(4, 8, 16, 26, torch.bfloat16)
    full = oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, Wb)
    ref = np.einsum("bhc,hec->bhe", run_oracle(c), Wb.to(torch.float64).numpy())
    assert np.array_equal(full, ref)
    pairs = [(1, 3), (0, 0), (1, 1)]
    got = oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, Wb, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(got[i], full[b, h])


def test_projection_multi_token_uses_each_heads_matrix():
    c, q = _multi(4, 2, 16, [6, 20], 2, seed=27)
    W_ = _proj_weights(4, 5, 16, 28)
    got = oracle.attention_proj(q, c.k, c.v, c.seq_lens, c.scale, W_)
    ref = np.einsum("bthc,hec->bthe", naive_causal_attention(q, c.k, c.v, c.seq_lens, c.scale),
                    widen(W_))
    assert got.shape == (2, 2, 4, 5)
    assert np.max(np.abs(got - ref)) <= 1e-13 * np.max(np.abs(ref))


def test_projection_negative_control_transposed_weights_are_caught():
    c = small(2, 1, 16, [25], seed=29)
    W_ = _proj_weights(2, 16, 16, 30)
    good = oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, W_)
    bad = oracle.attention_proj(c.q, c.k, c.v, c.seq_lens, c.scale, W_.transpose(1, 2))
    assert np.max(np.abs(good - bad)) > 1e-2
