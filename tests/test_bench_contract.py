"""The benchmark's reference arm keeps the JSON-line contract (CPU only).

`bench.py --impl reference` times the oracle on host cores. Its one JSON
line must carry the same metric, unit and direction as the GPU arm, the run's
step counts, a config naming the workload, a cpu_baseline that says how
many threads ran and what was sampled, and an e2e entry with no device copies.
"""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    sys.path.insert(0, ROOT)
    import bench
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--workload", "gqa8x2_f32_L4096"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "us/layer-step" and d["higher_is_better"] is False
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] >= 3
    assert d["value"] > 0 and abs(d["ms_per_step"] - d["value"] / 1e3) < 1e-2
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"] == "synthetic"
    c = d["config"]
    assert c["workload"] == "gqa8x2_f32_L4096" and c["seq_lens"] == [4096]
    assert (c["n_heads"], c["n_kv_heads"], c["head_dim"], c["kv_dtype"]) == (8, 2, 256, "f32")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "rows per step" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
