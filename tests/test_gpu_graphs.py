"""GPU parity of decode steps replayed from per-bucket CUDA graphs
(split_kv_decode_gb300.graphs.BucketedDecode): batch sizes and lengths change
from step to step, each step replays the graph of the smallest bucket that
holds the batch, and every active row is compared with the oracle."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from split_kv_decode_gb300 import workloads as W
from split_kv_decode_gb300.graphs import BucketedDecode, default_buckets
from tests.gpu_util import TOL, errors, oracle_rows

pytestmark = pytest.mark.gpu


def test_default_buckets():
    assert default_buckets(1) == [1]
    assert default_buckets(6) == [1, 2, 4, 6]
    assert default_buckets(8) == [1, 2, 4, 8]


STEPS = [[2500], [10, 3000, 777], [1, 2, 3, 2999, 1500, 64], [700, 1, 2048, 5, 3000]]


@pytest.mark.parametrize("hq,hkv,d,dtype,v_dim,mla", [
    (16, 4, 256, "f16", None, False),    # SIMT kernel
    (32, 1, 128, "bf16", None, False),   # tensor-core GQA kernel
    (32, 1, 576, "f32", 512, True),      # MLA kernels (f32 below 2048 positions, tensor cores above)
    (32, 2, 128, "f32", None, False),    # f32 CUDA-core kernel (16 rows per KV head)
])
def test_bucketed_graph_steps(hq, hkv, d, dtype, v_dim, mla):
    cap = 3000
    full = W.make_case("g", batch=6, n_heads=hq, n_kv_heads=hkv, head_dim=d, v_dim=v_dim,
                       seq_lens=[cap] * 6, kv_dtype=dtype, seed=1600 + hq,
                       scale=(1 / math.sqrt(576.0)) if mla else None, std=0.5 if mla else 1.0,
                       shared_kv=mla)
    q = torch.zeros(6, hq, d, device="cuda")
    k = full.k.cuda()
    v = k if mla else full.v.cuda()
    dec = BucketedDecode(q, k, v, full.scale, v_dim=v_dim)
    assert dec.buckets == [1, 2, 4, 6]
    g = torch.Generator().manual_seed(1601)
    for lens in STEPS:
        B = len(lens)
        qs = torch.randn((B, hq, d), generator=g)
        q[:B].copy_(qs)
        out = dec(lens)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        case = dataclasses.replace(full, batch=B, q=qs, k=full.k[:B], v=full.v[:B],
                                   seq_lens=torch.tensor(lens, dtype=torch.int32))
        worst, rel = errors(case, got, oracle_rows(case, threads=0))
        bar = TOL[dtype]
        assert np.all(np.isfinite(got)) and worst <= bar, (lens, worst, rel)
