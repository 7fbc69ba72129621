"""The bench's reference arm (the float64 oracle on the host cores) prints the
same one-line JSON contract as the CUDA arm: W warm-up rounds, then exactly K
timed rounds, with its own CPU baseline and an end-to-end figure that moves
no bytes between host and device.  Runs on the CPU (no GPU is touched)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "4", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "unit", "n_gpus", "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
                "data", "config"):
        assert key in d, key
    assert d["steps"] == 4 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tok/s" and d["higher_is_better"] is True
    assert abs(d["ms_per_step"] - 15 / d["value"] * 1e3) < 0.1 * d["ms_per_step"] + 0.1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]
