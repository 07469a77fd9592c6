"""The JSON line bench.py prints: the reference arm (the oracle timed on the
host cores, which needs no GPU) and our arm (a short run on the GPU), checked
key by key against the line's contract."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_line(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def check_common(d, steps, warmup):
    assert d["metric"].startswith("GEMM TFLOP/s")
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"].startswith("synthetic")
    names = [p["name"] for p in d["config"]["products"]]
    assert names == ["f32_4096_normal", "bf16_8192_normal"]
    assert "workload" in d["config"] and "l2" in d["config"]


def test_reference_arm_line():
    d = bench_line("--impl", "reference", "--steps", "2", "--warmup", "3",
                   "--reference-budget", "2")
    check_common(d, 2, 3)
    assert d["impl"] == "reference"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "seeded entries" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_our_arm_line():
    d = bench_line("--steps", "3", "--warmup", "3", "--no-cpu-baseline", timeout=900)
    check_common(d, 3, 3)
    assert d.get("impl", "ours") == "ours"
    r = d["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s" and r["workload"] == "f32_4096_normal"
    assert 0 < r["frac"] < 1.5 and abs(r["achieved"] / r["peak"] - r["frac"]) < 1e-3
    assert r["traffic"] is None or r["traffic"] > r["algorithmic_bytes"] / 2
    bf = d["rooflines"]["gemm_bf16f32"]
    assert bf["bound"] == "tensor" and 0 < bf["frac"] < 1.5
    per_call = d["gpu_launches_per_call"]
    assert set(per_call) == {"f32_4096_normal", "bf16_8192_normal"}
    assert all(isinstance(n, int) and n >= 1 for n in per_call.values()), per_call
    assert d["gpu_launches"] == 3 * sum(per_call.values())
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    assert c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)


@pytest.mark.gpu
def test_configs_line_reports_binding_and_graph_times():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--configs", "--steps", "5",
                        "--warmup", "3", "--shapes", "256x256x256:f32,512x512x512:bf16"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rows = json.loads(lines[0])["configs"]
    assert [row["entry"].split(" ")[0] for row in rows] == ["gemm_f32", "gemm_bf16f32"]
    for row in rows:
        assert row["ms"] > 0 and row["ms_graph"] is not None and row["ms_graph"] > 0
        assert row["frac_of_roofline_graph"] > 0
