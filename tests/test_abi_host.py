"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/split_kv_decode.h declares, its structs have the
C layout, the planner keeps its invariants, and bad arguments are refused
before anything touches a device."""
import ctypes
import math
import os
import re
import subprocess
import tempfile

import pytest

from split_kv_decode_gb300 import _native as N
from split_kv_decode_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "split_kv_decode.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(decode_attn_\w+)\s*\(",
                                 text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
        assert n in N.SIGNATURES, f"binding lacks {n}"



def test_every_exported_c_entry_point_is_declared(lib):
    # the reverse direction: the library exports no decode_attn_* function that
    # the header does not declare (nm lists the dynamic symbol table)
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines()
                       if l.split()[-1].startswith("decode_attn_")})
    assert exported == declared_functions()

def test_struct_layout_matches_the_c_compiler():
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "split_kv_decode.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n",
         sizeof(da_args_t), sizeof(da_plan_t),
         offsetof(da_args_t, k_batch_stride), offsetof(da_args_t, scale),
         offsetof(da_plan_t, seq_lens), offsetof(da_plan_t, workspace_bytes),
         offsetof(da_plan_t, est_cost), sizeof(da_dev_t), offsetof(da_dev_t, max_blocks_per_seq),
         offsetof(da_dev_t, num_blocks), offsetof(da_dev_t, v_block_stride),
         offsetof(da_args_t, q_len), sizeof(da_proj_t), offsetof(da_proj_t, out_dim),
         offsetof(da_proj_t, head_stride), offsetof(da_proj_t, row_stride));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "t")
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    want = [ctypes.sizeof(N.DaArgs), ctypes.sizeof(N.DaPlan), N.DaArgs.k_batch_stride.offset,
            N.DaArgs.scale.offset, N.DaPlan.seq_lens.offset, N.DaPlan.workspace_bytes.offset,
            N.DaPlan.est_cost.offset, ctypes.sizeof(N.DaDev), N.DaDev.max_blocks_per_seq.offset,
            N.DaDev.num_blocks.offset, N.DaDev.v_block_stride.offset, N.DaArgs.q_len.offset,
            ctypes.sizeof(N.DaProj), N.DaProj.out_dim.offset, N.DaProj.head_stride.offset,
            N.DaProj.row_stride.offset]
    assert got == want



def test_a_plain_c_program_plans_through_the_library(lib):
    """The boundary needs no Python: a C program built against the header and
    linked to libsplitkv.so plans the 151552-position 16/4-head workload, reads
    the workspace size, gets a refusal with a reason for 15 heads over 4 KV
    heads, and its plan equals the one the binding gets for the same arguments."""
    src = r"""
#include <stdio.h>
#include <string.h>
#include "split_kv_decode.h"
int main(void) {
  da_args_t a;
  static da_plan_t p;
  int32_t lens[1] = {151552};
  memset(&a, 0, sizeof a);
  a.batch = 1; a.n_heads = 16; a.n_kv_heads = 4; a.head_dim = 256; a.v_dim = 256;
  a.capacity = 151552;
  a.k_pos_stride = a.v_pos_stride = 4 * 256;
  a.k_head_stride = a.v_head_stride = 256;
  a.k_batch_stride = a.v_batch_stride = (int64_t)151552 * 4 * 256;
  a.kv_dtype = DA_F16; a.out_dtype = DA_F32; a.scale = 1.0f / 16;
  if (decode_attn_plan(&a, lens, 152, &p) != DA_OK) {
    printf("plan failed: %s\n", decode_attn_last_error());
    return 1;
  }
  printf("%d %d %d %d %d %d %lld %lld\n", p.kernel, p.tile, p.grid, p.n_items, p.n_splits[0],
         p.chunk[0], (long long)p.workspace_bytes, (long long)decode_attn_workspace_bytes(&p));
  a.n_heads = 15;
  int rc = decode_attn_plan(&a, lens, 152, &p);
  printf("%d\n", rc);
  printf("%s\n", decode_attn_last_error());
  printf("%s\n", decode_attn_version());
  return 0;
}
"""
    libdir = os.path.dirname(B.LIB)
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "plan.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "plan")
        subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        c, "-o", exe, "-L", libdir, "-lsplitkv", "-Wl,-rpath," + libdir],
                       check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    lines = out.splitlines()
    got = [int(x) for x in lines[0].split()]
    a = args(cap=151552)
    rc, p = plan(lib, a, [151552])
    assert rc == 0
    assert got == [p.kernel, p.tile, p.grid, p.n_items, p.n_splits[0], p.chunk[0],
                   p.workspace_bytes, p.workspace_bytes]
    assert int(lines[1]) == N.DA_EINVAL and "multiple" in lines[2]
    assert "sm_103a" in lines[3]


def args(batch=1, hq=16, hkv=4, d=256, dv=None, cap=262144, dt=N.DA_F16, out=N.DA_F32,
         force=0, layout="pos"):
    a = N.DaArgs()
    a.batch, a.n_heads, a.n_kv_heads, a.head_dim = batch, hq, hkv, d
    a.v_dim = d if dv is None else dv
    a.capacity = cap
    if layout == "pos":
        a.k_pos_stride = a.v_pos_stride = hkv * d
        a.k_head_stride = a.v_head_stride = d
    else:
        a.k_pos_stride = a.v_pos_stride = d
        a.k_head_stride = a.v_head_stride = cap * d
    a.k_batch_stride = a.v_batch_stride = cap * hkv * d
    a.kv_dtype, a.out_dtype = dt, out
    a.scale = 1.0 / math.sqrt(d)
    a.force_splits = force
    return a


def plan(lib, a, lens, sms=152):
    p = N.DaPlan()
    arr = (ctypes.c_int32 * len(lens))(*lens)
    rc = lib.decode_attn_plan(ctypes.byref(a), ctypes.cast(arr, ctypes.c_void_p), sms,
                              ctypes.byref(p))
    return rc, p


def check_invariants(a, p, lens, sms):
    G = a.n_heads // a.n_kv_heads
    assert p.batch == a.batch and p.kernel == N.DA_KERNEL_GQA_TMA
    base = 0
    for b, L in enumerate(lens):
        assert p.seq_lens[b] == L
        assert p.chunk[b] % p.tile == 0 and p.chunk[b] >= p.tile
        assert p.n_splits[b] == -(-L // p.chunk[b])                 # ceil
        assert (p.n_splits[b] - 1) * p.chunk[b] < L                  # no empty split
        assert p.split_base[b] == base
        base += p.n_splits[b]
    assert p.total_splits == base
    assert p.n_items == base * a.n_kv_heads
    assert 1 <= p.grid <= min(p.n_items, sms * p.ctas_per_sm)
    assert p.workspace_bytes >= base * a.n_heads * (a.v_dim + 2) * 4
    assert G * a.n_kv_heads == a.n_heads


@pytest.mark.parametrize("L", [1, 5, 33, 37, 64, 65, 4096, 4097, 8192, 12289, 20000, 151552,
                               262144])
def test_plan_invariants_single_sequence(lib, L):
    a = args()
    rc, p = plan(lib, a, [L])
    assert rc == 0, N.load().decode_attn_last_error()
    check_invariants(a, p, [L], 152)


def test_plan_fills_every_sm_at_long_context(lib):
    # 4 KV heads x splits >= 152 CTAs: the split budget is on the product
    for hkv, hq in ((4, 16), (2, 8), (8, 32), (1, 8)):
        a = args(hq=hq, hkv=hkv)
        rc, p = plan(lib, a, [151552])
        assert rc == 0
        assert p.grid >= 148                   # tile granularity may leave an SM or two idle
        # one balanced wave: makespan within 2% of the even share, plus one tile
        # of rounding and the modelled per-item cost (3 tiles)
        even = 151552 * hkv / 152
        assert p.est_cost <= even * 1.02 + 4 * p.tile


def test_plan_budget_follows_heads(lib):
    # fewer KV heads -> more splits per head (the "Attention at 128k" §5.1 trap)
    r8, p8 = plan(lib, args(hq=32, hkv=8), [65536])
    r2, p2 = plan(lib, args(hq=8, hkv=2), [65536])
    assert r8 == 0 and r2 == 0
    assert p2.n_splits[0] > p8.n_splits[0]
    assert p8.grid >= 148 and p2.grid >= 148


def cta_positions(p, lens, hkv):
    """Positions and items each CTA gets under the kernel's static round-robin
    (item i -> CTA i % grid; items ordered by sequence, split, then KV head)."""
    pos, items = [0] * p.grid, [0] * p.grid
    i = 0
    for b, L in enumerate(lens):
        for s in range(p.n_splits[b]):
            n = min(p.chunk[b], L - s * p.chunk[b])
            for _ in range(hkv):
                pos[i % p.grid] += n
                items[i % p.grid] += 1
                i += 1
    return pos, items


def test_plan_ragged_batch_is_balanced(lib):
    lens = [1024 + (i * 40961) % 130000 for i in range(32)]
    a = args(batch=32, hq=32, hkv=8, d=128, dt=N.DA_BF16, cap=max(lens))
    rc, p = plan(lib, a, lens)
    assert rc == 0
    check_invariants(a, p, lens, 152)
    pos, items = cta_positions(p, lens, 8)
    assert p.grid == 152
    assert max(pos) <= 1.05 * sum(pos) / len(pos)
    # per-sequence chunks keep the items few (each costs a merge) yet balanced
    assert max(items) <= 16


def test_plan_batch_of_equal_lengths_uses_one_chunk(lib):
    lens = [66000] * 32
    a = args(batch=32, hq=32, hkv=8, d=128, dt=N.DA_BF16, cap=66000)
    rc, p = plan(lib, a, lens)
    assert rc == 0
    check_invariants(a, p, lens, 152)
    assert len({p.chunk[b] for b in range(32)}) == 1
    pos, _ = cta_positions(p, lens, 8)
    assert max(pos) <= 1.03 * sum(pos) / len(pos)


def test_plan_forced_splits(lib):
    a = args(force=7)
    rc, p = plan(lib, a, [4097])
    assert rc == 0
    check_invariants(a, p, [4097], 152)
    assert p.n_splits[0] == 7
    a = args(force=1000)                      # capped so that no split is empty
    rc, p = plan(lib, a, [100])
    assert rc == 0 and p.n_splits[0] == -(-100 // p.tile)


def test_plan_small_sms_count(lib):
    a = args(batch=4, hq=24, hkv=4, dt=N.DA_F32, cap=131072)
    lens = [8192, 20480, 61440, 131072]
    for sms in (1, 7, 152):
        rc, p = plan(lib, a, lens, sms)
        assert rc == 0
        check_invariants(a, p, lens, sms)


@pytest.mark.parametrize("mutate,status", [
    (lambda a: setattr(a, "n_heads", 15), N.DA_EINVAL),
    (lambda a: setattr(a, "batch", 0), N.DA_EINVAL),
    (lambda a: setattr(a, "batch", 257), N.DA_EINVAL),
    (lambda a: setattr(a, "kv_dtype", 9), N.DA_EINVAL),
    (lambda a: setattr(a, "scale", float("nan")), N.DA_EINVAL),
    (lambda a: setattr(a, "k_pos_stride", 0), N.DA_EINVAL),
    (lambda a: setattr(a, "head_dim", 96) or setattr(a, "v_dim", 96), N.DA_EUNSUPPORTED),
    (lambda a: setattr(a, "v_dim", 128), N.DA_EUNSUPPORTED),
    (lambda a: setattr(a, "k_pos_stride", 1028), N.DA_EUNSUPPORTED),   # 2056 B: not 16-aligned
])
def test_plan_rejects_bad_arguments(lib, mutate, status):
    a = args()
    mutate(a)
    rc, _ = plan(lib, a, [4096])
    assert rc == status
    assert lib.decode_attn_last_error().decode()


def test_plan_rejects_bad_lengths(lib):
    a = args(cap=4096)
    assert plan(lib, a, [0])[0] == N.DA_EINVAL
    assert plan(lib, a, [4097])[0] == N.DA_EINVAL
    assert "seq_lens" in lib.decode_attn_last_error().decode()


def test_run_validates_before_launch(lib):
    a = args(cap=4096)
    rc, p = plan(lib, a, [4096])
    assert rc == 0
    P = ctypes.c_void_p
    fake = P(1 << 20)                        # never dereferenced: validation fails first
    rc = lib.decode_attn_splitk_ex(ctypes.byref(a), ctypes.byref(p), None, fake, fake, fake,
                                   fake, p.workspace_bytes, None)
    assert rc == N.DA_EINVAL
    rc = lib.decode_attn_splitk_ex(ctypes.byref(a), ctypes.byref(p), P(1 << 20 | 8), fake, fake,
                                   fake, fake, p.workspace_bytes, None)
    assert rc == N.DA_EINVAL                 # misaligned q
    rc = lib.decode_attn_splitk_ex(ctypes.byref(a), ctypes.byref(p), fake, fake, fake, fake,
                                   fake, p.workspace_bytes - 1, None)
    assert rc == N.DA_ENOSPACE
    p.n_splits[0] += 1                       # a tampered plan is refused
    rc = lib.decode_attn_splitk_ex(ctypes.byref(a), ctypes.byref(p), fake, fake, fake, fake,
                                   fake, p.workspace_bytes, None)
    assert rc == N.DA_EINVAL and "plan" in lib.decode_attn_last_error().decode()


def test_noalloc_refuses_a_split_only_call(lib):
    # with DA_FLAG_NO_COMBINE the partials would stay in the library's private
    # array, out of the caller's reach: the call is refused before any launch
    a = args(cap=4096)
    rc, p = plan(lib, a, [4096])
    assert rc == 0
    a.flags |= N.DA_FLAG_NO_COMBINE
    fake = ctypes.c_void_p(1 << 20)          # never dereferenced: validation fails first
    rc = lib.decode_attn_splitk_noalloc(ctypes.byref(a), ctypes.byref(p), fake, fake, fake,
                                        fake, None)
    assert rc == N.DA_EINVAL
    msg = lib.decode_attn_last_error().decode()
    assert "noalloc" in msg and "DA_FLAG_NO_COMBINE" in msg
    assert lib.decode_attn_splitk_noalloc(None, ctypes.byref(p), fake, fake, fake, fake,
                                          None) == N.DA_EINVAL


def test_version_and_null_handling(lib):
    assert b"sm_103a" in lib.decode_attn_version()
    assert lib.decode_attn_plan(None, None, 152, None) == N.DA_EINVAL
    assert lib.decode_attn_workspace_bytes(None) == 0
    assert lib.decode_attn_device_status(None, None) == N.DA_EINVAL


def mla_args(batch=1, hq=96, cap=131072, dt=N.DA_F32):
    a = N.DaArgs()
    a.batch, a.n_heads, a.n_kv_heads, a.head_dim, a.v_dim = batch, hq, 1, 576, 512
    a.capacity = cap
    a.k_pos_stride = a.v_pos_stride = 576
    a.k_head_stride = a.v_head_stride = 576
    a.k_batch_stride = a.v_batch_stride = cap * 576
    a.kv_dtype, a.out_dtype = dt, N.DA_F32
    a.scale = 1.0 / 24
    return a


def check_mla_invariants(a, p, lens, sms):
    assert p.kernel == N.DA_KERNEL_MLA_TC and p.tile == 16 and p.ctas_per_sm == 1
    base = 0
    for b, L in enumerate(lens):
        assert p.chunk[b] % 16 == 0
        assert p.n_splits[b] == -(-L // p.chunk[b]) and (p.n_splits[b] - 1) * p.chunk[b] < L
        assert p.split_base[b] == base
        base += p.n_splits[b]
    assert p.total_splits == base and p.n_items == base      # one KV head: item = split
    # a work item is one 2-CTA cluster: the grid is whole clusters, one CTA per SM
    assert p.grid % 2 == 0 and 2 <= p.grid <= 2 * p.n_items
    assert p.grid <= max(2, sms - sms % 2)
    assert p.workspace_bytes >= base * a.n_heads * (a.v_dim + 2) * 4


@pytest.mark.parametrize("hq,dt", [(32, N.DA_F32), (64, N.DA_F32), (96, N.DA_F32),
                                   (128, N.DA_F32), (96, N.DA_F16), (128, N.DA_BF16)])
def test_mla_plan_one_cluster_per_sm_pair(lib, hq, dt):
    a = mla_args(hq=hq, dt=dt)
    rc, p = plan(lib, a, [131072])
    assert rc == 0, lib.decode_attn_last_error()
    check_mla_invariants(a, p, [131072], 152)
    assert p.grid == 152 and p.n_items == 76        # one balanced wave of 76 clusters


@pytest.mark.parametrize("sms", [2, 3, 7, 148, 152])
def test_mla_plan_any_sm_count(lib, sms):
    lens = [700, 5000, 129, 131072]
    a = mla_args(batch=4)
    rc, p = plan(lib, a, lens, sms)
    assert rc == 0
    check_mla_invariants(a, p, lens, sms)


def test_mla_plan_short_context_and_forced_splits(lib):
    a = mla_args(cap=4096)
    for L in (1, 15, 16, 17, 4096):
        rc, p = plan(lib, a, [L])
        assert rc == 0
        check_mla_invariants(a, p, [L], 152)
    a.force_splits = 7
    rc, p = plan(lib, a, [2500])
    assert rc == 0 and p.n_splits[0] == 7
    check_mla_invariants(a, p, [2500], 152)


@pytest.mark.parametrize("mutate,msg", [
    (lambda a: setattr(a, "kv_dtype", N.DA_F16) or setattr(a, "flags", N.DA_FLAG_MLA_SIMT),
     "f32"),
    (lambda a: setattr(a, "n_heads", 48), "heads"),
    (lambda a: setattr(a, "n_heads", 160), "heads"),
    (lambda a: setattr(a, "k_pos_stride", 575) or setattr(a, "v_pos_stride", 575), "576"),
    (lambda a: setattr(a, "k_pos_stride", 577) or setattr(a, "v_pos_stride", 577), "aligned"),
    (lambda a: setattr(a, "v_pos_stride", 1152), "first 512"),
])
def test_mla_plan_rejects_unsupported_shapes(lib, mutate, msg):
    a = mla_args(cap=4096)
    mutate(a)
    rc, _ = plan(lib, a, [4096])
    assert rc == N.DA_EUNSUPPORTED
    assert msg in lib.decode_attn_last_error().decode()


def test_mla_run_needs_one_buffer_for_keys_and_values(lib):
    a = mla_args(cap=4096)
    rc, p = plan(lib, a, [4096])
    assert rc == 0
    P = ctypes.c_void_p
    fake, other = P(1 << 20), P(1 << 21)      # never dereferenced: validation fails first
    rc = lib.decode_attn_splitk_ex(ctypes.byref(a), ctypes.byref(p), fake, fake, other, fake,
                                   fake, p.workspace_bytes, None)
    assert rc == N.DA_EUNSUPPORTED
    assert "same buffer" in lib.decode_attn_last_error().decode()


def test_plan_cost_matches_a_per_item_simulation(lib):
    # est_cost is the makespan of the kernel's round-robin (item i -> CTA
    # i % grid) with a per-item cost of three tiles; replay it item by item
    import random
    rnd = random.Random(11)
    for _ in range(40):
        batch = rnd.randint(1, 40)
        hkv = rnd.choice([1, 2, 4, 8])
        lens = [rnd.randint(1, 200000) for _ in range(batch)]
        sms = rnd.choice([3, 76, 148, 152])
        a = args(batch=batch, hq=hkv * 4, hkv=hkv, d=128, dt=N.DA_BF16, cap=max(lens),
                 force=rnd.choice([0, 0, 0, 5]))
        rc, p = plan(lib, a, lens, sms)
        assert rc == 0
        check_invariants(a, p, lens, sms)
        pos, items = cta_positions(p, lens, hkv)
        assert p.est_cost == max(x + 3 * p.tile * n for x, n in zip(pos, items))


def test_plan_is_cheap_enough_for_every_decode_step(lib):
    import time
    lens = [1024 + (i * 40961) % 130000 for i in range(32)]
    a = args(batch=32, hq=32, hkv=8, d=128, dt=N.DA_BF16, cap=max(lens))
    p = N.DaPlan()
    arr = (ctypes.c_int32 * 32)(*lens)
    t0 = time.perf_counter()
    for _ in range(50):
        assert lib.decode_attn_plan(ctypes.byref(a), ctypes.cast(arr, ctypes.c_void_p), 152,
                                    ctypes.byref(p)) == 0
    per_plan = (time.perf_counter() - t0) / 50
    assert per_plan < 1e-3, per_plan


def paged_args(batch=2, hq=16, hkv=4, d=256, block_size=64, max_blocks=8, dt=N.DA_F16):
    a = args(batch=batch, hq=hq, hkv=hkv, d=d, dt=dt, cap=block_size * max_blocks)
    return a


def dev_struct(block_size=64, max_blocks=8, num_blocks=32, pos_stride=4 * 256, table=1 << 22,
               lens=1 << 23):
    d = N.DaDev()
    d.seq_lens = lens
    d.block_table = table
    d.max_blocks_per_seq, d.block_size, d.num_blocks = max_blocks, block_size, num_blocks
    d.k_block_stride = d.v_block_stride = block_size * pos_stride
    return d


@pytest.mark.parametrize("mutate,status,msg", [
    (lambda d: setattr(d, "block_size", 24), N.DA_EUNSUPPORTED, "multiple of 16"),
    (lambda d: setattr(d, "block_size", 0), N.DA_EUNSUPPORTED, "multiple of 16"),
    (lambda d: setattr(d, "num_blocks", 0), N.DA_EINVAL, "num_blocks"),
    (lambda d: setattr(d, "k_block_stride", 64 * 1024 - 8), N.DA_EUNSUPPORTED, "block strides"),
    (lambda d: setattr(d, "max_blocks_per_seq", 4), N.DA_EINVAL, "max_blocks_per_seq"),
    (lambda d: setattr(d, "block_table", (1 << 22) + 2), N.DA_EINVAL, "block_table"),
    (lambda d: setattr(d, "seq_lens", (1 << 23) + 1), N.DA_EINVAL, "seq_lens"),
])
def test_dev_call_validates_before_launch(lib, mutate, status, msg):
    a = paged_args()
    rc, p = plan(lib, a, [500, 300])
    assert rc == 0
    d = dev_struct()
    mutate(d)
    P = ctypes.c_void_p
    fake = P(1 << 20)                        # never dereferenced: validation fails first
    rc = lib.decode_attn_splitk_dev(ctypes.byref(a), ctypes.byref(p), ctypes.byref(d), fake,
                                    fake, fake, fake, fake, p.workspace_bytes, None)
    assert rc == status
    assert msg in lib.decode_attn_last_error().decode()


@pytest.mark.parametrize("hq,hkv,d,bs,kernel", [(32, 1, 128, 16, N.DA_KERNEL_GQA_TC),
                                                (16, 4, 256, 64, N.DA_KERNEL_GQA_TMA)])
def test_dev_call_paged_needs_chunks_on_the_box_grid(lib, hq, hkv, d, bs, kernel):
    # the GQA kernels copy a paged tile as boxes whose heights are multiples of
    # gcd(tile, block_size), starting at multiples of it, so a hand-made plan
    # whose chunk is off that grid is refused before any launch (the planner's
    # chunks are multiples of the tile)
    a = paged_args(hq=hq, hkv=hkv, d=d, block_size=bs, max_blocks=640 // bs)
    rc, p = plan(lib, a, [500, 300])
    assert rc == 0 and p.kernel == kernel
    h = math.gcd(p.tile, bs)
    assert all(p.chunk[b] % p.tile == 0 for b in range(2)) and h < p.tile
    L, n = 500, p.n_splits[0]
    c = next(c for c in range(p.chunk[0], 0, -1) if c % h and -(-L // c) == n)
    p.chunk[0] = c
    P = ctypes.c_void_p
    fake = P(1 << 20)
    d = dev_struct(block_size=bs, max_blocks=640 // bs, num_blocks=100, pos_stride=hkv * d)
    rc = lib.decode_attn_splitk_dev(ctypes.byref(a), ctypes.byref(p), ctypes.byref(d), fake,
                                    fake, fake, fake, fake, p.workspace_bytes, None)
    assert rc == N.DA_EINVAL and "multiples of %d" % h in lib.decode_attn_last_error().decode()


def test_dev_call_needs_one_latent_pool_for_mla_and_an_extension(lib):
    a = mla_args(cap=4096)
    rc, p = plan(lib, a, [4096])
    assert rc == 0
    P = ctypes.c_void_p
    fake, other = P(1 << 20), P(1 << 21)
    d = dev_struct(block_size=64, max_blocks=64, pos_stride=576)
    d.v_block_stride = d.k_block_stride + 576 * 4
    rc = lib.decode_attn_splitk_dev(ctypes.byref(a), ctypes.byref(p), ctypes.byref(d), fake,
                                    fake, fake, fake, fake, p.workspace_bytes, None)
    assert rc == N.DA_EUNSUPPORTED and "one pool" in lib.decode_attn_last_error().decode()
    d = dev_struct(block_size=64, max_blocks=64, pos_stride=576)
    rc = lib.decode_attn_splitk_dev(ctypes.byref(a), ctypes.byref(p), ctypes.byref(d), fake,
                                    fake, other, fake, fake, p.workspace_bytes, None)
    assert rc == N.DA_EUNSUPPORTED and "same buffer" in lib.decode_attn_last_error().decode()
    a = paged_args()
    rc, p = plan(lib, a, [500, 300])
    rc = lib.decode_attn_splitk_dev(ctypes.byref(a), ctypes.byref(p), None, fake, fake, fake,
                                    fake, fake, p.workspace_bytes, None)
    assert rc == N.DA_EINVAL


# ---------------------------------------------------------------------------
# several query tokens per sequence (q_len > 1)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("hq,hkv,q_len", [(16, 4, 2), (8, 4, 4), (4, 4, 6), (4, 4, 8), (32, 8, 2)])
def test_plan_multi_token_groups(lib, hq, hkv, q_len):
    d = 128 if hq == 32 else 256
    a = args(hq=hq, hkv=hkv, d=d, cap=8192)
    rc, p1 = plan(lib, a, [8192])
    assert rc == 0
    a.q_len = q_len
    rc, p = plan(lib, a, [8192])
    assert rc == 0, lib.decode_attn_last_error().decode()
    # the workspace holds q_len rows per head for every split
    ml = p.total_splits * hq * q_len * 8
    acc = p.total_splits * hq * q_len * a.v_dim * 4
    assert p.workspace_bytes >= ml + acc
    # 8 or more rows per item on a 16-bit cache go to the tensor-core kernel
    rows = hq // hkv * q_len
    assert p.kernel == (N.DA_KERNEL_GQA_TC if rows >= 8 else N.DA_KERNEL_GQA_TMA)


@pytest.mark.parametrize("hq,hkv,q_len,dt", [(64, 1, 4, N.DA_F16), (128, 1, 2, N.DA_BF16),
                                             (64, 1, 3, N.DA_F32)])
def test_plan_multi_token_rejects_large_groups(lib, hq, hkv, q_len, dt):
    # more than 128 rows per work item: no kernel holds them
    a = args(hq=hq, hkv=hkv, cap=8192, dt=dt)
    a.q_len = q_len
    rc, _ = plan(lib, a, [8192])
    assert rc == N.DA_EUNSUPPORTED
    assert "q_len" in lib.decode_attn_last_error().decode()


@pytest.mark.parametrize("hq,hkv,q_len,d,per", [(16, 4, 3, 256, 6), (8, 2, 4, 256, 8),
                                                (16, 1, 2, 128, 8), (24, 4, 2, 256, 6),
                                                (32, 1, 1, 128, 8), (64, 2, 4, 128, 8),
                                                (11, 1, 1, 128, 1), (27, 1, 1, 256, 3)])
def test_plan_f32_cache_with_many_rows_takes_simt_row_groups(lib, hq, hkv, q_len, d, per):
    # 9 to 128 rows per (sequence, KV head) on an f32 cache: the SIMT kernel
    # with the rows cut into groups of the largest divisor up to 8, one work
    # item per (sequence, KV head, split, row group)
    a = args(hq=hq, hkv=hkv, d=d, cap=65536, dt=N.DA_F32)
    a.q_len = q_len
    rows = hq // hkv * q_len
    rc, p = plan(lib, a, [65536], 152)
    assert rc == 0, lib.decode_attn_last_error()
    assert p.kernel == N.DA_KERNEL_GQA_TMA
    assert p.n_items == p.total_splits * hkv * (rows // per)
    assert p.chunk[0] % p.tile == 0


@pytest.mark.parametrize("hq,hkv,q_len,d,dt", [(32, 1, 1, 128, N.DA_F16), (16, 4, 4, 256, N.DA_BF16),
                                               (64, 1, 2, 256, N.DA_F16), (8, 1, 1, 256, N.DA_BF16),
                                               (16, 2, 8, 128, N.DA_F16)])
def test_plan_tensor_core_gqa(lib, hq, hkv, q_len, d, dt):
    a = args(batch=3, hq=hq, hkv=hkv, d=d, cap=20000, dt=dt)
    a.q_len = q_len
    lens = [q_len, 777, 20000]
    rc, p = plan(lib, a, lens)
    assert rc == 0, lib.decode_attn_last_error().decode()
    tile = 64                               # positions per tile
    assert p.kernel == N.DA_KERNEL_GQA_TC and p.tile == tile and p.ctas_per_sm == 1
    base = 0
    for b, L in enumerate(lens):
        assert p.chunk[b] % tile == 0 and p.n_splits[b] == -(-L // p.chunk[b])
        assert p.split_base[b] == base
        base += p.n_splits[b]
    assert p.n_items == base * hkv and 1 <= p.grid <= min(152, p.n_items)


def test_plan_simt_flag_keeps_eight_row_groups_on_the_simt_kernel(lib):
    a = args(hq=8, hkv=1, d=256, cap=4096, dt=N.DA_F16)
    assert plan(lib, a, [4096])[1].kernel == N.DA_KERNEL_GQA_TC
    a.flags = N.DA_FLAG_GQA_SIMT
    assert plan(lib, a, [4096])[1].kernel == N.DA_KERNEL_GQA_TMA
    a = args(hq=16, hkv=1, d=256, cap=4096, dt=N.DA_F16)  # 16 rows: tensor cores only
    a.flags = N.DA_FLAG_GQA_SIMT
    assert plan(lib, a, [4096])[1].kernel == N.DA_KERNEL_GQA_TC


def test_plan_multi_token_needs_q_len_positions(lib):
    a = args(hq=8, hkv=4, cap=8192)
    a.q_len = 4
    assert plan(lib, a, [4, 100])[0] == 0
    assert plan(lib, a, [3, 100])[0] == N.DA_EINVAL
    assert "q_len" in lib.decode_attn_last_error().decode()
    a.q_len = -1
    assert plan(lib, a, [100])[0] == N.DA_EINVAL
    a.q_len = 0                                # 0 reads as one token
    assert plan(lib, a, [1])[0] == 0


@pytest.mark.parametrize("hq,q_len,ok", [(48, 2, True), (16, 4, True), (32, 3, True),
                                         (16, 6, True), (64, 2, True), (32, 4, True),
                                         (96, 2, False), (24, 2, False)])
def test_mla_multi_token_rows(lib, hq, q_len, ok):
    # the rows of an MLA item are (token, head) pairs: 32, 64 or 96 of them
    a = mla_args(hq=hq, cap=4096)
    a.q_len = q_len
    rc, p = plan(lib, a, [4096])
    if ok:
        assert rc == 0 and p.kernel == N.DA_KERNEL_MLA_TC
        assert p.workspace_bytes >= p.total_splits * hq * q_len * (512 * 4 + 8)
    else:
        assert rc == N.DA_EUNSUPPORTED
        assert "rows" in lib.decode_attn_last_error().decode()


# ---------------------------------------------------------------------------
# the combine fused with a per-head projection: validation before any launch
# ---------------------------------------------------------------------------
def _proj(w=1 << 20, dt=N.DA_F32, out_dim=128, hs=0, rs=0):
    p = N.DaProj()
    p.w, p.w_dtype, p.out_dim, p.head_stride, p.row_stride = w, dt, out_dim, hs, rs
    return p


@pytest.mark.parametrize("proj,status,msg", [
    (_proj(w=0), N.DA_EINVAL, "NULL"),
    (_proj(dt=N.DA_F16), N.DA_EUNSUPPORTED, "f32 or bf16"),
    (_proj(out_dim=0), N.DA_EUNSUPPORTED, "out_dim"),
    (_proj(out_dim=257), N.DA_EUNSUPPORTED, "out_dim"),
    (_proj(w=(1 << 20) | 8), N.DA_EINVAL, "aligned"),
    (_proj(rs=258), N.DA_EINVAL, "aligned"),            # 1032 B rows: not a 16-byte multiple
    (_proj(rs=128), N.DA_EINVAL, "row_stride"),
    (_proj(dt=N.DA_BF16, hs=4), N.DA_EINVAL, "aligned"),
])
def test_combine_proj_validates_weights(lib, proj, status, msg):
    a = args(cap=4096)
    rc, p = plan(lib, a, [4096])
    assert rc == 0
    P = ctypes.c_void_p
    fake = P(1 << 21)                        # never dereferenced: validation fails first
    rc = lib.decode_attn_combine_proj(ctypes.byref(a), ctypes.byref(p), ctypes.byref(proj),
                                      fake, 1, fake, None)
    assert rc == status
    assert msg in lib.decode_attn_last_error().decode()
    rc = lib.decode_attn_splitk_proj(ctypes.byref(a), ctypes.byref(p), ctypes.byref(proj), fake,
                                     fake, fake, fake, fake, p.workspace_bytes, None)
    assert rc == status



@pytest.mark.parametrize("hq,hkv,d,dt", [(12, 4, 256, N.DA_F32), (40, 8, 128, N.DA_BF16),
                                         (14, 2, 256, N.DA_F16), (15, 5, 128, N.DA_F16)])
def test_plan_odd_groups_on_the_simt_kernel(lib, hq, hkv, d, dt):
    # groups of 3, 5 and 7 heads per KV head (e.g. 40 query / 8 KV heads)
    a = args(hq=hq, hkv=hkv, d=d, cap=8192, dt=dt)
    rc, p = plan(lib, a, [8192])
    assert rc == 0, lib.decode_attn_last_error().decode()
    assert p.kernel == N.DA_KERNEL_GQA_TMA
    check_invariants(a, p, [8192], 152)


# ---------------------------------------------------------------------------
# a seeded sweep over every kernel's shapes
# ---------------------------------------------------------------------------
def _random_shape(rnd):
    """(kind, args, lens, sms) for one random shape that the planner must accept."""
    kind = rnd.choice(["simt", "tc", "mla"])
    batch = rnd.choice([1, 1, 2, 3, 4, 7, 16, 32, 64, 128, 256])
    if kind == "mla":
        hq, q_len = rnd.choice([(96, 1), (64, 1), (32, 1), (48, 2), (32, 2), (32, 3), (16, 4)])
        cap = rnd.choice([64, 4096, 131072, 262144])
        a = mla_args(batch=batch, hq=hq, cap=cap)
        hkv = 1
    else:
        hkv = rnd.choice([1, 2, 4, 8])
        d = rnd.choice([128, 256])
        if kind == "simt":
            dt = rnd.choice([N.DA_F32, N.DA_F16, N.DA_BF16])
            rows = rnd.randint(1, 8)
        else:
            dt = rnd.choice([N.DA_F16, N.DA_BF16])
            rows = rnd.randint(8, 128)
        # rows per item = heads per KV head x new tokens
        q_len = rnd.choice([q for q in range(1, min(rows, 64) + 1) if rows % q == 0])
        gh = rows // q_len
        cap = rnd.choice([64, 4096, 131072, 262144])
        a = args(batch=batch, hq=gh * hkv, hkv=hkv, d=d, dt=dt, cap=cap,
                 layout=rnd.choice(["pos", "head"]))
        if kind == "simt" and rows == 8 and dt != N.DA_F32:
            a.flags = N.DA_FLAG_GQA_SIMT          # 8 rows on a 16-bit cache stay on SIMT
    a.q_len = q_len
    if rnd.random() < 0.2:
        a.force_splits = rnd.randint(1, 400)
    short = rnd.random() < 0.3
    lens = [rnd.randint(q_len, min(cap, 300) if short else cap) for _ in range(batch)]
    sms = rnd.choice([1, 2, 3, 7, 76, 132, 148, 151, 152])
    return kind, hkv, a, lens, sms


def test_plan_random_shapes_on_every_kernel(lib):
    """600 seeded shapes across the three split kernels (batch 1-256, 1-8 KV
    heads, 1-64 new tokens, both cache layouts, 1-152 SMs, forced splits now
    and then). Every plan must cover each sequence with non-empty splits of
    whole tiles, keep its totals consistent with its tables, launch whole
    clusters within the SMs it was given, and size a workspace that holds
    every partial and stays 256-byte aligned when ranks are stacked."""
    import random
    rnd = random.Random(2024)
    want_kernel = {"simt": N.DA_KERNEL_GQA_TMA, "tc": N.DA_KERNEL_GQA_TC,
                   "mla": N.DA_KERNEL_MLA_TC}
    for case in range(600):
        kind, hkv, a, lens, sms = _random_shape(rnd)
        rc, p = plan(lib, a, lens, sms)
        where = f"case {case}: {kind} batch {a.batch} hq {a.n_heads} hkv {hkv} q_len {a.q_len} " \
                f"sms {sms} force {a.force_splits}"
        assert rc == 0, f"{where}: {lib.decode_attn_last_error().decode()}"
        assert p.kernel == want_kernel[kind], where
        assert p.batch == a.batch and p.tile >= 1, where
        if kind == "tc":
            assert p.tile == 64, where
        if kind == "mla":
            assert p.tile == 16, where
        base = 0
        for b, L in enumerate(lens):
            c = p.chunk[b]
            assert p.seq_lens[b] == L and c >= p.tile and c % p.tile == 0, where
            assert p.n_splits[b] == -(-L // c) and (p.n_splits[b] - 1) * c < L, where
            if a.force_splits:
                assert p.n_splits[b] <= a.force_splits, where
            assert p.split_base[b] == base, where
            base += p.n_splits[b]
        assert p.total_splits == base and p.n_items == base * hkv, where
        cluster = 2 if kind == "mla" else 1
        assert p.grid % cluster == 0 and cluster <= p.grid <= p.n_items * cluster, where
        per_sm = max(cluster, (sms * p.ctas_per_sm) // cluster * cluster)
        assert p.grid <= per_sm, where
        rows = a.n_heads * a.q_len
        partials = base * rows * (a.v_dim + 2) * 4
        counters = max(2, a.batch * hkv) * 4      # arrival counters of the one-launch merge
        assert lib.decode_attn_workspace_bytes(ctypes.byref(p)) == p.workspace_bytes, where
        assert partials + counters <= p.workspace_bytes <= partials + counters + 1024, where
        assert p.workspace_bytes % 256 == 0, where


def test_plans_and_error_messages_are_per_thread(lib):
    """decode_attn_plan is pure host code and its failure message is
    thread-local: eight threads planning at once (ctypes releases the GIL for
    the call), half of them with a bad head count, each get the plan a lone
    call gets and only their own message."""
    import threading
    lens = [151552, 4096, 20000, 77777]
    want = {}
    for i, L in enumerate(lens):
        rc, p = plan(lib, args(cap=262144), [L])
        assert rc == 0
        want[i] = (p.n_splits[0], p.chunk[0], p.grid, p.workspace_bytes)
    errors, results = [], {}

    def worker(t):
        try:
            for it in range(200):
                i = (t + it) % len(lens)
                a = args(cap=262144)
                if t % 2:
                    a.n_heads = 15 + 2 * (t % 3)          # 15, 17 or 19 over 4 KV heads
                    rc, _ = plan(lib, a, [lens[i]])
                    msg = lib.decode_attn_last_error().decode()
                    if rc != N.DA_EINVAL or f"n_heads {a.n_heads} " not in msg:
                        errors.append((t, rc, msg))
                else:
                    rc, p = plan(lib, a, [lens[i]])
                    got = (p.n_splits[0], p.chunk[0], p.grid, p.workspace_bytes)
                    if rc != 0 or got != want[i]:
                        errors.append((t, rc, got, want[i]))
            results[t] = True
        except Exception as e:                          # pragma: no cover
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors[:5]
    assert len(results) == 8


def test_header_constants_match_the_binding():
    # every #define of the header that the binding mirrors has the same value
    text = open(HEADER).read()
    defs = dict(re.findall(r"^#define\s+(DA_\w+)\s+(0x[0-9a-fA-F]+|\d+)", text, flags=re.M))
    mirrored = [k for k in defs if hasattr(N, k)]
    assert len(mirrored) >= 10
    for k in mirrored:
        assert getattr(N, k) == int(defs[k], 0), k


def test_mla_kernel_flags_exclude_each_other(lib):
    a = mla_args(cap=4096)
    a.flags = N.DA_FLAG_MLA_SIMT | N.DA_FLAG_MLA_TC
    rc, _ = plan(lib, a, [1000])
    assert rc == N.DA_EINVAL and "exclude" in lib.decode_attn_last_error().decode()


@pytest.mark.parametrize("hq", [32, 64, 96])
def test_mla_short_sequences_plan_for_the_f32_kernel(lib, hq):
    # every sequence below DA_MLA_EXACT_BELOW: the f32 kernel runs one CTA per
    # (item, group of 32 rows), so the items fill the SMs divided by the groups
    a = mla_args(hq=hq, cap=4096)
    groups = hq // 32
    for L in (1, 100, 1000, N.DA_MLA_EXACT_BELOW - 1):
        rc, p = plan(lib, a, [L], 152)
        assert rc == 0
        check_mla_invariants(a, p, [L], 152)
        assert p.n_items <= max(1, 152 // groups) or p.n_splits[0] * 16 >= L
    # at the threshold the tensor-core kernel's geometry: one item per SM pair
    rc, p = plan(lib, a, [4096], 152)
    assert rc == 0 and p.n_items <= 76 * 4
