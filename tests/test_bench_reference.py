"""bench.py --impl reference: the oracle timed on the host prints one JSON line
with the GPU arm's metric, unit and direction; under torchrun only rank 0
prints; a long prefill chunk is sampled by query so the arm stays short."""

import json
import os
import subprocess
import sys

import bench
from libbuild import ROOT


def _run(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_the_contract_line():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == bench.DEFAULT_WORKLOAD
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_timed_queries_sample_long_chunks_only():
    assert bench.timed_queries(bench.Scenario("gqa_decode", 0)) == (None, 1.0)
    assert bench.timed_queries(bench.Scenario("gqa_verify4", 0)) == (None, 1.0)
    js, frac = bench.timed_queries(bench.Scenario("gqa_prefill512", 0))
    assert len(js) == 16 and 0 in js and 511 in js
    assert frac == 16 / 512


def test_all_cores_oracle_timing_runs_processes_together():
    sc = bench.Scenario("gqa_decode", 0)
    r = bench.cpu_baseline_all_cores(sc, 0.5, 2)
    assert r["cores"] == 2 and r["value"] > 0
    assert "2 processes" in r["sample"]
