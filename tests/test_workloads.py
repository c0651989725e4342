"""The seeded input recipe (CPU only).

Both the oracle and the kernels are fed by split_kv_decode_gb300.workloads, so
its recipe is checked on its own: the same seed gives the same bits, the named
workloads have the geometries, storage types, scales and spreads of the pages'
workloads, positions past a sequence's length are NaN (so an unmasked read
shows), and the ragged batch's lengths are drawn uniform in [1024, 131072].
"""
import math

import numpy as np
import torch

from split_kv_decode_gb300 import workloads as W


def test_same_seed_same_bits_other_seed_other_bits():
    kw = dict(batch=2, n_heads=8, n_kv_heads=2, head_dim=64, seq_lens=[300, 200],
              kv_dtype="bf16")
    a, b = W.make_case("a", seed=5, **kw), W.make_case("b", seed=5, **kw)
    c = W.make_case("c", seed=6, **kw)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
    assert not torch.equal(a.q, c.q)
    assert not torch.equal(a.k[0, :200].float(), c.k[0, :200].float())


def test_tails_past_each_length_are_nan_and_the_rest_finite():
    c = W.make_case("t", batch=3, n_heads=4, n_kv_heads=2, head_dim=32, seq_lens=[10, 64, 1],
                    kv_dtype="f16", capacity=64)
    for b, L in enumerate(c.seq_lens.tolist()):
        assert torch.isfinite(c.k[b, :L].float()).all() and torch.isfinite(c.v[b, :L].float()).all()
        assert torch.isnan(c.k[b, L:].float()).all() and torch.isnan(c.v[b, L:].float()).all()


def test_named_geometries_types_and_scales():
    want = {
        "gqa_8x2": (1, 8, 2, 256, 256, "f32", "f32", 1 / 16, [4096]),
        "gqa_16x4": (1, 16, 4, 256, 256, "f16", "f32", 1 / 16, [151552]),
        "mla_96": (1, 96, 1, 576, 512, "f32", "f32", 1 / 24, [131072]),
        "gqa_24x4": (4, 24, 4, 256, 256, "f32", "f32", 1 / 16, list(W.GQA24X4_LENS)),
        "ragged_32": (32, 32, 8, 128, 128, "bf16", "bf16", 1 / math.sqrt(128),
                      W.ragged_lens(1238)),
    }
    for name, (B, hq, hkv, dk, dv, kvt, outt, scale, lens) in want.items():
        c = W.named(name, scale_lens=1 / 256)      # small lengths; the geometry is the same
        assert (c.batch, c.n_heads, c.n_kv_heads, c.head_dim, c.v_dim) == (B, hq, hkv, dk, dv)
        assert (c.kv_dtype, c.out_dtype) == (kvt, outt)
        assert abs(c.scale - scale) < 1e-15
        assert c.seq_lens.tolist() == [max(1, round(x / 256)) for x in lens]
        assert c.q.dtype == torch.float32 and c.q.shape == (B, hq, dk)
        assert c.shared_kv == (name == "mla_96")
        if c.shared_kv:
            assert c.v is c.k                      # values are the first 512 columns of K
    assert W.GQA16X4_RUNGS == (4096, 20480, 61440, 151552, 262144)


def test_ragged_lengths_are_uniform_in_range_and_seeded():
    lens = W.ragged_lens(1238)
    assert len(lens) == 32 and lens == W.ragged_lens(1238)
    assert all(1024 <= x <= 131072 for x in lens)
    many = np.array(W.ragged_lens(99, batch=20000))
    assert many.min() >= 1024 and many.max() <= 131072
    # uniform: mean and spread of U[1024, 131072] within sampling error
    mu, sd = (1024 + 131072) / 2, (131072 - 1024) / math.sqrt(12)
    assert abs(many.mean() - mu) < 4 * sd / math.sqrt(many.size)
    assert abs(many.std() - sd) < 0.02 * sd


def test_value_spreads_follow_the_recipe():
    # N(0, 1) for the GQA caches and q; N(0, 0.5^2) for the MLA latent
    g = W.make_case("t", batch=1, n_heads=4, n_kv_heads=2, head_dim=256, seq_lens=[4000])
    m = W.named("mla_96", scale_lens=1 / 64)
    for x, sd in ((g.k[0], 1.0), (g.v[0], 1.0), (g.q, 1.0), (m.k[0, :2048], 0.5)):
        x = x.double()
        n = x.numel()
        assert abs(float(x.mean())) < 5 * sd / math.sqrt(n)
        assert abs(float(x.std()) - sd) < 0.01 * sd


def test_multi_token_queries_are_seeded_and_shaped():
    a, b = W.multi_token_q(2, 4, 16, 256, seed=3), W.multi_token_q(2, 4, 16, 256, seed=3)
    assert a.shape == (2, 4, 16, 256) and a.dtype == torch.float32 and torch.equal(a, b)
    assert not torch.equal(a, W.multi_token_q(2, 4, 16, 256, seed=4))
