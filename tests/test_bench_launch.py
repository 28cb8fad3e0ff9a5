"""bench.py's own launcher and reporting helpers on the CPU: `--gpus 2` outside torchrun starts two
ranks (gloo here) that agree on the max-over-ranks time; the median interval; the oracle timing
leg (one core, then one spawned process per row group)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpus_2_starts_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--launch-check",
                        "--steps", "50"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{") and "launch_check" in ln]
    assert len(lines) == 1                          # rank 0 alone prints
    d = lines[0]
    assert d["world"] == 2 and d["ranks"] == [0, 1] and d["backend"] == "gloo"
    assert d["max_ms"] == 15.0                      # rank 1's 15 ms, not rank 0's 10 ms
    assert d["tokens_per_s"] == pytest.approx(2 * 6 * 50 / 0.015)


def test_median_interval():
    import bench
    r = bench.median_ci([1.0] * 10 + [2.0] * 21)
    assert r["median"] == 2.0 and r["n"] == 31
    assert r["ci95"][0] <= r["median"] <= r["ci95"][1]
    c = bench.median_ci([3.0] * 30)
    assert c["ci95"] == [3.0, 3.0]


def test_cpu_identity_fields():
    import bench
    c = bench.cpu_identity()
    assert c["nproc"] >= 1 and 1 <= c["affinity"] <= c["nproc"] and c["model"]


def test_oracle_timing_legs_on_the_tiny_layer():
    import bench
    r = bench.run_oracle_child("tiny", 4, steps=1, warmup=0, one_core_steps=1)
    assert r["rows"] == 4 and r["one_core"]["cores"] == 1 and r["one_core"]["value"] > 0
    if r["cpu"]["affinity"] > 1:
        assert r["all_cores"]["cores"] == 4 and r["all_cores"]["value"] > 0
    line = bench.cpu_baseline_line(r, "tiny", 4, extrapolated=False)
    assert line["kind"] == "oracle" and line["unit"] == "tokens/s"
    assert line["value"] == max(v["value"] for v in (line["one_core"], line["all_cores"] or line["one_core"]))
