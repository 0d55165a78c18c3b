"""The reference arm of bench.py (the CPU oracle timed as it stands) keeps the
bench contract: one JSON line on rank 0 with the decode metric, a time-like
value, the oracle described as the CPU baseline and an end-to-end object with
no host-device traffic; other ranks print nothing and exit 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(rank: int):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2" if rank else "1")
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                          capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)


def test_reference_arm_prints_one_contract_line():
    res = run_reference(0)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "us/layer" and d["higher_is_better"] is False
    assert d["value"] > 0 and abs(d["ms_per_step"] - d["value"] / 1000.0) < 1e-9
    assert d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["data"] == "synthetic" and d["config"]["batch"] == 1 and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work():
    res = run_reference(1)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""
