"""Benchmark: decode-attention µs per layer-step and KV GB/s on GB300.

A step is one decode token through one attention layer for every sequence of
the workload: the host plan, the split kernel and the combine kernel, called
through the library's C ABI. Default workload: 16 query / 4 KV heads,
head_dim 256, f16 KV cache, f32 q, context 151552 (the Qwen3.5-9B-like
geometry at its rung nearest 128k; 620.8 MB of K+V per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-extra]

Timing: W untimed warm-up steps (plus a short soak so the clocks settle);
then K steps, each bracketed by CUDA events on the launching stream around
its launches (the step's host plan is made first, while the L2 flush -- a
write of 2 x L2 bytes, then a read of 2 x L2 bytes so that the write's dirty
lines are written back before the step, all outside the events -- runs on the
GPU); barrier + synchronize on both sides; max over ranks. The default run
adds `configs`: the same measurement, over 100 steps, for every workload of
the pages' configurations. `--impl reference` times the double-precision CPU
oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: (named case, seq_len override[, new tokens per sequence])
    "gqa16x4_f16_L151552": ("gqa_16x4", 151552),
    "gqa16x4_f16_L262144": ("gqa_16x4", 262144),
    "gqa16x4_f16_L61440": ("gqa_16x4", 61440),
    "gqa16x4_f16_L20480": ("gqa_16x4", 20480),
    "gqa16x4_f16_L4096": ("gqa_16x4", 4096),
    "gqa8x2_f32_L4096": ("gqa_8x2", None),
    "gqa24x4_f32_b4": ("gqa_24x4", None),
    "ragged32_bf16": ("ragged_32", None),
    "mla96_f32_L131072": ("mla_96", None),
    "mla128_f32_L131072": ("mla_128", None),
    "mla96_f16_L131072": ("mla_96_f16", None),
    # four new tokens per sequence on the default cache: 16 query rows per KV head
    "gqa16x4_f16_L151552_q4": ("gqa_16x4", 151552, 4),
    # two new tokens on the 27B-like f32 cache: 12 rows per KV head (f32 kernel)
    "gqa24x4_f32_b4_q2": ("gqa_24x4", None, 2),
}
DEFAULT = "gqa16x4_f16_L151552"
METRIC = "decode-attention us/layer-step (and KV GB/s)"   # both arms report this metric
# the split kernel each workload runs, and the arithmetic type it computes in
KERNEL = {"mla96_f32_L131072": ("mla_split_kernel", "bf16"),
          "mla128_f32_L131072": ("mla_split_kernel", "bf16"),
          "mla96_f16_L131072": ("mla_split_kernel", "f16"),
          "gqa16x4_f16_L151552_q4": ("gqa_tc_kernel", "f16")}
DEFAULT_KERNEL = ("gqa_split_kernel", "f32")


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the default process group (x itself
    on a single rank): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s, no MEASURED_PEAKS.json)"


KERNEL_SOURCES = {
    "gqa_split_kernel": ("gqa_split.cuh", "gqa_inst.cuh", "gqa_f32.cu", "gqa_f16.cu", "gqa_bf16.cu",
                         "merge.cuh"),
    "gqa_tc_kernel": ("gqa_tc.cu", "gqa_split.cuh", "merge.cuh"),
    "mla_split_kernel": ("mla_split.cu", "merge.cuh"),
    "f32_split_kernel": ("f32_split.cu",),
}


def kernel_source_hash(kernel):
    """Hash of the sources a split kernel is compiled from (its own files plus
    the shared PTX helpers and internal header)."""
    import hashlib
    h = hashlib.sha256()
    src = os.path.join(ROOT, "split_kv_decode_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel] + ("ptx.cuh", "internal.h"):
        h.update(open(os.path.join(src, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_file(kernel, workload):
    return os.path.join(ROOT, "profiles", f"{kernel.replace('_kernel', '')}_{workload}.traffic.txt")


def profiled_traffic(kernel, workload):
    """Per-launch DRAM bytes of the split kernel from the committed ncu summary,
    or None if there is none for this workload or the kernel changed since."""
    try:
        lines = open(traffic_file(kernel, workload)).read().splitlines()
    except OSError:
        return None
    kv = dict(l.split(":", 1) for l in lines if ":" in l and not l.startswith("#"))
    kv = {k.strip(): v.strip() for k, v in kv.items()}
    if kv.get("workload") != workload or kv.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return int(float(kv["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        mhz = statistics.median(r[0] for r in rows)
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for n, v in zip(names, r[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": mhz, "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def make_inputs(workload, device, draw_on_device=False, scale_lens=1.0):
    """The workload's seeded case on `device`. With several new tokens per
    sequence, case.q is [B, q_len, Hq, Dk]. draw_on_device: draw the caches on
    `device` (same recipe, other values; for timing only). scale_lens shrinks
    every length (a smaller case of the same workload, for profiler captures)."""
    import dataclasses
    from split_kv_decode_gb300 import workloads as W
    name, L = WORKLOADS[workload][:2]
    q_len = WORKLOADS[workload][2] if len(WORKLOADS[workload]) > 2 else 1
    where = str(device) if draw_on_device else "cpu"
    case = (W.named(name, seq_len=L, device=where, scale_lens=scale_lens) if L else
            W.named(name, device=where, scale_lens=scale_lens))
    if q_len > 1:
        case = dataclasses.replace(case, q=W.multi_token_q(case.batch, q_len, case.n_heads,
                                                           case.head_dim))
    q = case.q.to(device)
    k = case.k.to(device)
    v = k if case.shared_kv else case.v.to(device)
    return case, q, k, v


def out_shape(case):
    return tuple(case.q.shape[:-1]) + (case.v_dim,)


def oracle_rows(case, pairs, threads):
    """The oracle on the (b, h) rows `pairs` (every new token of them)."""
    import oracle
    fn = oracle.attention_multi if case.q.dim() == 4 else oracle.attention
    return fn(case.q, case.k, case.v, case.seq_lens, case.scale, v_dim=case.v_dim, pairs=pairs,
              threads=threads)


def cpu_baseline(case, budget_s=12.0):
    """Time the oracle (as it stands) on all host cores over a bounded sample of
    the workload: whole (b, h) rows at full context, repeated until about
    budget_s seconds of wall time, scaled to one full layer-step."""
    import oracle
    threads = oracle.max_threads()
    pairs_all = [(b, h) for b in range(case.batch) for h in range(case.n_heads)]
    t0 = time.perf_counter()
    oracle_rows(case, [pairs_all[0]], 1)
    t_row = time.perf_counter() - t0
    # rows per repetition: all of them, or as many as fit in a third of the budget
    n = max(1, min(len(pairs_all), int(budget_s / 3 / max(t_row, 1e-6) * threads)))
    stride = max(1, len(pairs_all) // n)
    pairs = pairs_all[::stride][:n]
    pos_sample = sum(int(case.seq_lens[b]) for b, _ in pairs)
    pos_all = sum(int(case.seq_lens[b]) for b, _ in pairs_all)
    times, t_start = [], time.perf_counter()
    while not times or (time.perf_counter() - t_start < budget_s and len(times) < 50):
        t0 = time.perf_counter()
        oracle_rows(case, pairs, threads)
        times.append(time.perf_counter() - t0)
    us = statistics.median(times) * 1e6 * pos_all / pos_sample
    pos_row = int(case.seq_lens[pairs_all[0][0]])
    return {"value": round(us, 1), "unit": "us/layer-step", "cores": threads, "kind": "oracle",
            "single_thread": {"value": round(t_row * 1e6 * pos_all / pos_row, 1),
                              "sample": "one (b,h) row at full context on one thread, scaled"},
            "sample": f"{len(pairs)} of {len(pairs_all)} (b,h) rows at full context, median of "
                      f"{len(times)} repetitions ({time.perf_counter() - t_start:.1f} s), "
                      "scaled by attended positions"}


def run_reference(args, budget_s=150.0):
    """The reference arm: the CPU oracle, timed on host cores, rank 0 only.

    Each step times a bounded sample of the workload, sized from --steps and
    --warmup so that the whole run takes about budget_s seconds of host work:
    whole (b, h) rows while one row fits a step's share, else one row per core
    over a prefix of each sampled sequence's context. The oracle's time per row
    is linear in the attended positions, so every step is scaled to the full
    layer-step by attended positions."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    case, _, _, _ = make_inputs(args.workload, "cpu")
    import oracle
    threads = oracle.max_threads()
    pairs_all = [(b, h) for b in range(case.batch) for h in range(case.n_heads)]
    pos_all = sum(int(case.seq_lens[b]) for b, _ in pairs_all)
    t0 = time.perf_counter()
    oracle_rows(case, [pairs_all[0]], 1)
    t_row = max(time.perf_counter() - t0, 1e-6)               # one full row, one thread
    per_step = min(2.0, max(0.02, budget_s / (args.steps + args.warmup)))
    if t_row <= per_step:
        n = max(1, min(len(pairs_all), int(per_step / t_row) * threads))
        frac = 1.0
    else:
        n = min(len(pairs_all), threads)
        frac = per_step / t_row
    stride = max(1, len(pairs_all) // n)
    pairs = pairs_all[::stride][:n]
    q_len = int(case.q.shape[1]) if case.q.dim() == 4 else 1
    lens = case.seq_lens.clone()
    if frac < 1.0:
        for b in range(case.batch):
            L = int(case.seq_lens[b])
            lens[b] = min(L, max(q_len, 64, int(math.ceil(L * frac))))
    sample = dataclasses.replace(case, seq_lens=lens)
    pos_sample = sum(int(lens[b]) for b, _ in pairs)
    for _ in range(args.warmup):
        oracle_rows(sample, pairs[:1], threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_rows(sample, pairs, threads)
        times.append((time.perf_counter() - t0) * pos_all / pos_sample)
    us = statistics.mean(times) * 1e6
    what = "full context" if frac >= 1.0 else \
        f"the first {frac:.1%} of each sampled sequence's positions"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1),
        "unit": "us/layer-step", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, case),
        "cpu_baseline": {"value": round(us, 1), "unit": "us/layer-step", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{len(pairs)} of {len(pairs_all)} (b,h) rows per step at "
                                   f"{what}, scaled by attended positions"},
        "e2e": {"value": round(us, 1), "unit": "us/layer-step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(workload, case):
    return {"workload": workload, "batch": case.batch, "n_heads": case.n_heads,
            "n_kv_heads": case.n_kv_heads, "head_dim": case.head_dim, "v_dim": case.v_dim,
            "seq_lens": (case.seq_lens.tolist() if case.batch <= 8 else
                         f"{case.batch} lengths, sum {int(case.seq_lens.sum())}"),
            "q_len": int(case.q.shape[1]) if case.q.dim() == 4 else 1,
            "kv_dtype": case.kv_dtype, "q_dtype": "f32", "out_dtype": case.out_dtype,
            "kv_bytes_per_step": case.kv_bytes, "parallelism": "replicas",
            "l2": "flushed between steps (2 x L2 write, then 2 x L2 read so no dirty line of the flush is written back in the step; outside the events)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the e2e and cpu_baseline measurements")
    ap.add_argument("--no-soak", action="store_true",
                    help="skip the clock soak (for profiler runs, which serialise launches)")
    ap.add_argument("--scale-lens", type=float, default=1.0,
                    help="shrink every length by this factor (smaller profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    from split_kv_decode_gb300 import api as A
    from split_kv_decode_gb300 import _native as N

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    case, q, k, v = make_inputs(args.workload, dev, scale_lens=args.scale_lens)
    out_dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[case.out_dtype]
    stream = torch.cuda.current_stream(dev)

    # a step: one call, which runs the split kernel and the combine; for
    # comparison, the split kernel alone (DA_FLAG_NO_COMBINE) and the one-launch
    # form (DA_FLAG_ONE_LAUNCH)
    a_step = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
    a_split = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt,
                          flags=N.DA_FLAG_NO_COMBINE)
    plan = A.decode_attn_plan(a_step, case.seq_lens.tolist())
    ws = torch.empty(A.decode_attn_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    out = torch.empty(out_shape(case), dtype=out_dt, device=dev)
    lens = case.seq_lens.tolist()
    flush = L2Flush(dev)
    launches = count_launches(a_step, plan)

    def make_plan():
        return A.decode_attn_plan(a_step, lens)         # host plan (no sync)

    def run_step(p):
        A.decode_attn_splitk_ex(a_step, p, q, k, v, out, ws, stream)

    def split(p):
        A.decode_attn_splitk_ex(a_split, p, q, k, v, out, ws, stream)
        return p

    for _ in range(args.warmup):
        run_step(make_plan())
    torch.cuda.synchronize()
    # clocks are sampled from here on: a short untimed soak brings them under
    # load, then the timed steps run; every sample is taken with the GPU busy
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + (0.0 if args.no_soak else 0.6)
    while time.time() < t_end:
        for _ in range(20):
            run_step(make_plan())
        torch.cuda.synchronize()
    # the timed steps: events only around the whole step, so the combine's
    # programmatic launch overlaps the split kernel's tail as it does in use
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        # each step plans on the host while the flush runs on the GPU, so the
        # events bracket the device work of the step, not host scheduling
        p = make_plan()
        flush(i)
        ev[i][0].record(stream)
        run_step(p)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    # the split kernel alone, without the merge (DA_FLAG_NO_COMBINE), for
    # comparison; L2 flushed before each
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        p = make_plan()
        flush(i)
        evs[i][0].record(stream)
        split(p)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    clocks["window"] = "untimed soak (0.6 s) + timed steps + split-only steps"
    if world > 1:
        dist.barrier()
    A.decode_attn_device_status(ws, stream)

    step_us = [ev[i][0].elapsed_time(ev[i][1]) * 1e3 for i in range(args.steps)]
    one_us = None if args.no_extra else time_one_launch(case, q, k, v, out_dt, dev, flush, args)
    split_us = [evs[i][0].elapsed_time(evs[i][1]) * 1e3 for i in range(args.steps)]
    # value: the median step (max over ranks), which a few steps slowed by the
    # clock sampler's queries do not move; the mean and every step beside it
    value = max_over_ranks(statistics.median(step_us), dev)
    step_mean = max_over_ranks(statistics.mean(step_us), dev)
    split_mean = statistics.mean(split_us)
    peak, peak_src = load_peaks()
    # the dominant kernel: the split kernel (with one launch per step, the step
    # itself)
    kernel_us = statistics.mean(step_us) if launches == 1 else split_mean
    achieved = case.kv_bytes / (kernel_us * 1e-6) / 1e9
    kv_gbs_step = case.kv_bytes / (value * 1e-6) / 1e9
    kernel, arith = KERNEL.get(args.workload, DEFAULT_KERNEL)

    line = {
        "metric": METRIC, "value": round(value, 2),
        "unit": "us/layer-step", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": arith, "data": "synthetic",
        "config": workload_config(args.workload, case),
        "kv_gbs": round(kv_gbs_step, 1),
        "hbm_frac_of_8tbs": round(kv_gbs_step / 8000.0, 4),
        "value_statistic": "median of the timed steps (max over ranks)",
        "step_us_mean": round(step_mean, 2),
        "step_us_all": [round(x, 1) for x in step_us[:64]],
        "launches_per_step": launches,
        "one_launch_step_us_median": one_us,
        "split_only_us_median": round(statistics.median(split_us), 2),
        "plan": {"grid": plan.grid, "items": plan.n_items, "tile": plan.tile,
                 "chunk": plan.chunk[0], "n_splits": plan.n_splits[0]},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(kernel, args.workload),
                     "kernel": kernel, "peak_source": peak_src,
                     "kernel_us_mean": round(kernel_us, 2),
                     "what": ("split kernel merging its own partials (the whole step, one launch)"
                              if launches == 1 else "split kernel (a combine launch follows)"),
                     "bytes_per_launch": case.kv_bytes},
        "clocks": clocks,
        "gpu_launches": launches * args.steps,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if rank == 0 and not args.no_extra:
        line["configs"] = measure_configs(dev, peak)
        line["e2e"] = measure_e2e(case, q, out_dt, dev, stream, args)
        line["hot_l2"] = measure_hot(case, q, k, v, out_dt, dev, args)
        line["copy_probe"] = read_probe(dev, stream, max(case.kv_bytes, 512 << 20))
        if kernel == "gqa_split_kernel" and case.q.dim() == 3:
            line["graph"] = measure_graph(case, q, k, v, out_dt, dev, flush, args)
            line["paged"] = {f"block_{bs}": measure_paged(case, q, k, v, out_dt, dev, flush, args, bs)
                             for bs in (16, 64, 256)}
            ml = measure_multi_token(case, k, v, out_dt, dev, flush, args)
            if ml:
                line["multi_token"] = ml
        if kernel == "mla_split_kernel":
            line["wv_b"] = {name: measure_wv_b(case, q, k, v, out_dt, dev, flush, args, wdt)
                            for name, wdt in (("f32", torch.float32), ("bf16", torch.bfloat16))}
        line["cpu_baseline"] = cpu_baseline(case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def count_launches(a, p):
    """Kernel launches of one decode_attn_splitk_ex call with args `a` and plan
    `p`: the split kernel(s) -- for the MLA shape the tensor-core kernel and/or
    the f32 kernel, by the lengths -- and the combine, unless the split kernel
    merges its own partials (DA_FLAG_ONE_LAUNCH). Mirrors the library's rules
    (documented in its header); the counter memset of the one-launch form is not
    a kernel of ours and is not counted."""
    from split_kv_decode_gb300 import _native as N
    if p.kernel != N.DA_KERNEL_MLA_TC:
        split, exact = 1, False
    else:
        below = (1 << 31) if a.flags & N.DA_FLAG_MLA_SIMT else (
            0 if a.flags & N.DA_FLAG_MLA_TC else N.DA_MLA_EXACT_BELOW)
        lens = [p.seq_lens[b] for b in range(p.batch)]
        exact = any(L < below for L in lens)
        split = int(any(L >= below for L in lens)) + int(exact)
    if a.flags & N.DA_FLAG_NO_COMBINE:
        return split
    fused = bool(a.flags & N.DA_FLAG_ONE_LAUNCH) and not exact
    return split + (0 if fused else 1)


def time_one_launch(case, q, k, v, out_dt, dev, flush, args):
    """Median step time with the merge folded into the split kernel
    (DA_FLAG_ONE_LAUNCH), for comparison with the default two launches."""
    import torch
    from split_kv_decode_gb300 import _native as N
    from split_kv_decode_gb300 import api as A
    a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt,
                    flags=N.DA_FLAG_ONE_LAUNCH)
    lens = case.seq_lens.tolist()
    p = A.decode_attn_plan(a, lens)
    ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
    out = torch.empty(out_shape(case), dtype=out_dt, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        A.decode_attn_splitk_ex(a, A.decode_attn_plan(a, lens), q, k, v, out, ws, stream)
    us = _timed_steps(lambda: A.decode_attn_splitk_ex(a, p, q, k, v, out, ws, stream), flush,
                      max(20, min(args.steps, 200)), stream)
    return round(us, 2)


# every workload the pages' configurations name, in the default run
CONFIG_SWEEP = ("gqa8x2_f32_L4096", "gqa16x4_f16_L4096", "gqa16x4_f16_L20480",
                "gqa16x4_f16_L61440", "gqa16x4_f16_L151552", "gqa16x4_f16_L262144",
                "mla96_f32_L131072", "gqa24x4_f32_b4", "ragged32_bf16", "gqa16x4_f16_L151552_q4",
                "mla128_f32_L131072", "mla96_f16_L131072", "gqa24x4_f32_b4_q2")


def time_split_and_step(workload, dev, steps):
    """Step (split + combine) and split-kernel times of one workload, each over
    `steps` runs with the L2 flushed before every run (CUDA events on the
    launching stream; the host plan is made before the flush). The caches are
    drawn on the device (same recipe as the parity cases, other values)."""
    import torch
    from split_kv_decode_gb300 import _native as N
    from split_kv_decode_gb300 import api as A
    case, q, k, v = make_inputs(workload, dev, draw_on_device=True)
    out_dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[case.out_dtype]
    stream = torch.cuda.current_stream(dev)
    a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
    a_split = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt,
                          flags=N.DA_FLAG_NO_COMBINE)
    lens = case.seq_lens.tolist()
    p0 = A.decode_attn_plan(a, lens)
    ws = torch.empty(A.decode_attn_workspace_bytes(p0), dtype=torch.uint8, device=dev)
    out = torch.empty(out_shape(case), dtype=out_dt, device=dev)
    flush = L2Flush(dev)
    for _ in range(3):
        A.decode_attn_splitk_ex(a, A.decode_attn_plan(a, lens), q, k, v, out, ws, stream)
    torch.cuda.synchronize()
    st, sp = [], []
    for i in range(steps):
        p = A.decode_attn_plan(a, lens)
        flush(i)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        A.decode_attn_splitk_ex(a, p, q, k, v, out, ws, stream)
        e[1].record(stream)
        st.append(e)
    for i in range(steps):
        p = A.decode_attn_plan(a_split, lens)
        flush(i)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        A.decode_attn_splitk_ex(a_split, p, q, k, v, out, ws, stream)
        e[1].record(stream)
        sp.append(e)
    a_one = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt,
                        flags=N.DA_FLAG_ONE_LAUNCH)
    for _ in range(3):
        A.decode_attn_splitk_ex(a_one, A.decode_attn_plan(a_one, lens), q, k, v, out, ws, stream)
    p1 = A.decode_attn_plan(a_one, lens)
    one_us = _timed_steps(lambda: A.decode_attn_splitk_ex(a_one, p1, q, k, v, out, ws, stream),
                          flush, max(20, steps // 2), stream)
    torch.cuda.synchronize()
    A.decode_attn_device_status(ws, stream)
    step_us = [x.elapsed_time(y) * 1e3 for x, y in st]
    split_us = [x.elapsed_time(y) * 1e3 for x, y in sp]
    kernel = {N.DA_KERNEL_GQA_TMA: "gqa_split_kernel", N.DA_KERNEL_GQA_TC: "gqa_tc_kernel",
              N.DA_KERNEL_MLA_TC: "mla_split_kernel"}.get(p0.kernel, str(p0.kernel))
    res = (case, kernel, step_us, split_us, p0, count_launches(a, p0), one_us)
    del q, k, v, ws, out, flush
    torch.cuda.empty_cache()
    return res


def measure_configs(dev, peak, steps=100):
    """Every configuration of the sweep: step and split-kernel times (mean and
    median), KV GB/s per step, and the split kernel's fraction of the measured
    HBM bandwidth."""
    res = {}
    for w in CONFIG_SWEEP:
        case, kernel, step_us, split_us, p, launches, one_us = time_split_and_step(w, dev, steps)
        sm = statistics.mean(split_us)
        km = statistics.mean(step_us) if launches == 1 else sm
        res[w] = {
            "kernel": kernel, "kv_bytes": case.kv_bytes, "steps": steps,
            "launches_per_step": launches,
            "step_us_mean": round(statistics.mean(step_us), 2),
            "step_us_median": round(statistics.median(step_us), 2),
            "split_only_us_mean": round(sm, 2),
            "split_only_us_median": round(statistics.median(split_us), 2),
            "one_launch_step_us_median": round(one_us, 2),
            "kv_gbs": round(case.kv_bytes / (statistics.mean(step_us) * 1e-6) / 1e9, 1),
            "kernel_frac_of_measured_hbm": round(case.kv_bytes / (km * 1e-6) / 1e9 / peak, 4),
            "splits": p.n_splits[0], "items": p.n_items, "grid": p.grid,
        }
    return res


class L2Flush:
    """The L2 flush between timed steps: a write of a buffer twice the L2's size,
    then a read of another such buffer. The read evicts the lines the write left
    dirty, so their write-back to HBM happens here and not inside the next timed
    step: the timed work starts on an L2 of clean, unrelated lines (the state a
    profiler's cache control gives, and the one a decode step meets after kernels
    that mostly read weights). None of the step's inputs is in L2 either way."""

    def __init__(self, dev):
        import torch
        n = 2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4 + 1024
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self(0) # the first call pays torch's one-time host work, outside any timed loop
        torch.cuda.synchronize(dev)

    def __call__(self, i):
        import torch
        self.w.fill_(float(i))
        torch.sum(self.r, dim=0, out=self.sink)


def _timed_steps(launch, flush, steps, stream):
    """Median CUDA-event time (us) of `launch` over `steps` runs, L2 flushed before each."""
    import torch
    ts = []
    for i in range(steps):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) * 1e3 for a, b in ts)


def measure_graph(case, q, k, v, out_dt, dev, flush, args):
    """The step (split + combine) through decode_attn_splitk_dev with the lengths
    in device memory, captured once in a CUDA graph and replayed: no host work
    per step."""
    import torch
    from split_kv_decode_gb300 import api as A
    a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
    out = torch.empty(case.batch, case.n_heads, case.v_dim, dtype=out_dt, device=dev)
    dev_lens = case.seq_lens.to(dev)
    d = A.make_dev(seq_lens=dev_lens)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for _ in range(3):
            A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, s)
    n = max(20, min(args.steps, 200))
    with torch.cuda.stream(s):
        us = _timed_steps(g.replay, flush, n, s)
    return {"value": round(us, 2), "unit": "us/layer-step", "steps": n,
            "what": "whole step replayed from one CUDA graph, lengths read on the device"}


def measure_paged(case, q, k, v, out_dt, dev, flush, args, block_size):
    """The same step with the caches scattered into pools of `block_size`-position
    blocks in a random order, read through a block table (decode_attn_splitk_dev).
    A tile is copied as boxes of gcd(tile, block_size) rows, each inside one
    block, so tiles stay whole at any block size."""
    import torch
    from split_kv_decode_gb300 import api as A
    B, cap, hkv, dk = k.shape
    nb = -(-cap // block_size)
    num_blocks = B * nb
    order = torch.randperm(num_blocks, generator=torch.Generator().manual_seed(5)).to(dev)
    table = order.view(B, nb).to(torch.int32).contiguous()
    kp = torch.empty(num_blocks, block_size, hkv, dk, dtype=k.dtype, device=dev)
    vp = torch.empty(num_blocks, block_size, hkv, v.shape[3], dtype=v.dtype, device=dev)
    pad = nb * block_size - cap
    kpad = torch.nn.functional.pad(k, (0, 0, 0, 0, 0, pad)) if pad else k
    vpad = torch.nn.functional.pad(v, (0, 0, 0, 0, 0, pad)) if pad else v
    kp[table.view(-1).long()] = kpad.reshape(B * nb, block_size, hkv, dk)
    vp[table.view(-1).long()] = vpad.reshape(B * nb, block_size, hkv, v.shape[3])
    del kpad, vpad
    a = A.make_paged_args(q, kp, vp, case.scale, nb, out_dtype=out_dt)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
    out = torch.empty(case.batch, case.n_heads, case.v_dim, dtype=out_dt, device=dev)
    d = A.make_dev(block_table=table, k_pool=kp, v_pool=vp)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        A.decode_attn_splitk_dev(a, p, d, q, kp, vp, out, ws, stream)
    n = max(20, min(args.steps, 200))
    us = _timed_steps(lambda: A.decode_attn_splitk_dev(a, p, d, q, kp, vp, out, ws, stream),
                      flush, n, stream)
    gbs = case.kv_bytes / (us * 1e-6) / 1e9
    del kp, vp
    torch.cuda.empty_cache()
    return {"value": round(us, 2), "unit": "us/layer-step", "steps": n, "block_size": block_size,
            "kv_gbs": round(gbs, 1),
            "what": "whole step with the caches in a pool of blocks, random block order"}


def measure_wv_b(case, q, k, v, out_dt, dev, flush, args, wdt):
    """The step with the value up-projection wv_b fused into the combine: every
    head's merged 512-wide latent times its [128 x 512] matrix (random weights
    of that shape), split + combine_proj."""
    import torch
    from split_kv_decode_gb300 import api as A
    g = torch.Generator().manual_seed(77)
    w = (torch.randn((case.n_heads, 128, case.v_dim), generator=g) / 23.0).to(wdt).to(dev)
    a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
    out = torch.empty(case.batch, case.n_heads, 128, dtype=out_dt, device=dev)
    pj = A.make_proj(w)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        A.decode_attn_splitk_proj(a, p, pj, q, k, v, out, ws, stream)
    n = max(20, min(args.steps, 200))
    us = _timed_steps(lambda: A.decode_attn_splitk_proj(a, p, pj, q, k, v, out, ws, stream),
                      flush, n, stream)
    return {"value": round(us, 2), "unit": "us/layer-step", "steps": n,
            "w_bytes": w.numel() * w.element_size(),
            "what": f"split + combine fused with wv_b ({case.n_heads} x 128 x {case.v_dim} "
                    f"{str(wdt).split('.')[-1]} weights)"}


def measure_multi_token(case, k, v, out_dt, dev, flush, args):
    """The same caches with q_len = 2, 4, 8 new tokens per sequence (causal among
    themselves): every K/V tile is read once for all of them. Query rows per KV
    head (heads per KV head x q_len) of 8 to 128 run on the tensor-core kernel
    (16-bit caches); the SIMT kernel takes up to 8 rows."""
    import torch
    from split_kv_decode_gb300 import api as A
    from split_kv_decode_gb300 import _native as N
    from split_kv_decode_gb300 import workloads as W
    G = case.n_heads // case.n_kv_heads
    res = {}
    for q_len in (2, 4, 8):
        rows = G * q_len
        if int(case.seq_lens.min()) < q_len:
            continue
        if not (rows <= 8 or (case.kv_dtype in ("f16", "bf16") and rows <= 128)):
            continue
        q = W.multi_token_q(case.batch, q_len, case.n_heads, case.head_dim).to(dev)
        a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
        p = A.decode_attn_plan(a, case.seq_lens.tolist())
        ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
        out = torch.empty(case.batch, q_len, case.n_heads, case.v_dim, dtype=out_dt, device=dev)
        stream = torch.cuda.current_stream(dev)
        for _ in range(3):
            A.decode_attn_splitk_ex(a, p, q, k, v, out, ws, stream)
        n = max(20, min(args.steps, 200))
        us = _timed_steps(lambda: A.decode_attn_splitk_ex(a, p, q, k, v, out, ws, stream),
                          flush, n, stream)
        res[f"q_len_{q_len}"] = {
            "value": round(us, 2), "unit": "us/layer-step", "steps": n, "rows_per_item": rows,
            "kernel": "gqa_tc_kernel" if p.kernel == N.DA_KERNEL_GQA_TC else "gqa_split_kernel",
            "kv_gbs": round(case.kv_bytes / (us * 1e-6) / 1e9, 1)}
    if not res:
        return None
    res["what"] = ("whole step for q_len new tokens per sequence, causal among "
                   "themselves, sharing every K/V tile")
    return res


def measure_hot(case, q, k, v, out_dt, dev, args, reps=10):
    """The step with no L2 flush between steps (labelled: inputs that fit the
    129 MB L2 are then served from it). The device time alone: `reps`
    consecutive steps (with the lengths read on the device) are captured in one
    CUDA graph and replayed, so host work does not show."""
    import torch
    from split_kv_decode_gb300 import api as A
    a = A.make_args(q, k, v, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
    p = A.decode_attn_plan(a, case.seq_lens.tolist())
    ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
    out = torch.empty(out_shape(case), dtype=out_dt, device=dev)
    d = A.make_dev(seq_lens=case.seq_lens.to(device=dev, dtype=torch.int32))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))

    def one():
        A.decode_attn_splitk_dev(a, p, d, q, k, v, out, ws, s)

    with torch.cuda.stream(s):
        for _ in range(3):
            one()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                one()
    torch.cuda.synchronize()
    ts = []
    with torch.cuda.stream(s):                    # replay() launches on the current stream
        g.replay()
        for _ in range(max(5, min(args.steps, 50))):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            ts.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(x.elapsed_time(y) * 1e3 for x, y in ts) / reps
    return {"value": round(us, 2), "unit": "us/layer-step", "steps": len(ts) * reps,
            "what": f"whole step, {reps} steps per CUDA graph replay, no L2 flush",
            "fits_l2": case.kv_bytes < 120 * (1 << 20)}


def read_probe(dev, stream, nbytes):
    """An in-run bandwidth probe beside the measured copy peak: torch's copy of a
    buffer of at least the workload's K/V bytes (read + write bytes / time; L2
    flushed before each copy), to show the state of this box during the run."""
    import torch
    x = torch.ones(nbytes // 2, dtype=torch.float16, device=dev)
    y = torch.empty_like(x)
    flush = L2Flush(dev)
    ts = []
    for i in range(13):
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        y.copy_(x)
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ts[3:])
    del x, y, flush
    torch.cuda.empty_cache()
    return {"gbs": round(2 * nbytes / (us * 1e-6) / 1e9, 1), "bytes_copied": nbytes,
            "what": "torch copy_ of an f16 buffer (read + write bytes), L2 flushed before each"}


def measure_e2e(case, q_dev, out_dt, dev, stream, args):
    """The same step through the public API with host buffers: per step the
    inputs (q and the K/V cache) are copied from pinned host memory, the call
    runs, and the output is copied back; all inside the events."""
    import torch
    from split_kv_decode_gb300 import api as A
    hq = case.q.pin_memory()
    hk = case.k.pin_memory()
    hv = hk if case.shared_kv else case.v.pin_memory()
    hout = torch.empty(out_shape(case), dtype=out_dt).pin_memory()
    dq = torch.empty_like(hq, device=dev)
    dk = torch.empty_like(hk, device=dev)
    dv = dk if case.shared_kv else torch.empty_like(hv, device=dev)
    dout = torch.empty(hout.shape, dtype=out_dt, device=dev)
    lens = case.seq_lens.tolist()
    a = A.make_args(dq, dk, dv, case.scale, v_dim=case.v_dim, out_dtype=out_dt)
    p = A.decode_attn_plan(a, lens)
    ws = torch.empty(A.decode_attn_workspace_bytes(p), dtype=torch.uint8, device=dev)
    n = max(3, min(args.steps, 20))

    def once():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        if not case.shared_kv:
            dv.copy_(hv, non_blocking=True)
        pp = A.decode_attn_plan(a, lens)
        A.decode_attn_splitk_ex(a, pp, dq, dk, dv, dout, ws, stream)
        hout.copy_(dout, non_blocking=True)

    for _ in range(2):
        once()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        once()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    h2d = hq.numel() * hq.element_size() + hk.numel() * hk.element_size() + (
        0 if case.shared_kv else hv.numel() * hv.element_size())
    d2h = hout.numel() * hout.element_size()
    # the cache-resident variant: only q in and out back per step
    e0.record(stream)
    for _ in range(n):
        dq.copy_(hq, non_blocking=True)
        pp = A.decode_attn_plan(a, lens)
        A.decode_attn_splitk_ex(a, pp, dq, dk, dv, dout, ws, stream)
        hout.copy_(dout, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    us_res = e0.elapsed_time(e1) * 1e3 / n
    return {"value": round(us, 1), "unit": "us/layer-step", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n,
            "cache_resident": {"value": round(us_res, 2), "unit": "us/layer-step",
                               "h2d_bytes_per_step": hq.numel() * hq.element_size(),
                               "d2h_bytes_per_step": d2h}}


if __name__ == "__main__":
    sys.exit(main())
