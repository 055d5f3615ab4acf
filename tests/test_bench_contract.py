"""The reference arm of bench.py (the CPU oracle timed on the host cores) runs
without a GPU and prints one JSON line with the keys the benchmark contract
names; its metric, unit and workload are the GPU arm's."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("flag,metric,name", [(None, bench.METRIC, "cp_chunks"),
                                              ("--bwd", bench.BWD_METRIC, "cp_chunks"),
                                              ("--indexer", bench.IDX_METRIC, "indexer_cp")])
def test_reference_arm_json_line(flag, metric, name):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1"]
    out = subprocess.run(cmd + ([flag] if flag else []), cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout[-2000:]
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["metric"] == metric and rec["unit"] == bench.UNIT
    assert rec["value"] > 0 and rec["higher_is_better"] is True
    assert rec["n_gpus"] == 1 and rec["steps"] == 2 and rec["warmup"] >= 3
    assert rec["ms_per_step"] > 0
    assert rec["config"]["name"] == name and "workload" in rec["config"]
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == rec["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = rec["e2e"]
    assert e2e["value"] == rec["value"] and e2e["unit"] == rec["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
