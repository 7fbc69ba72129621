"""The bench's command line on the CPU: the library drives one GPU, so a
multi-GPU request prints a one-line record and exits without touching a
GPU; the reference arm's ranks other than 0 exit quietly."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, **env):
    e = dict(os.environ, **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=e, capture_output=True,
                          text=True, timeout=120)


def test_multi_gpu_request_is_a_one_line_record():
    r = _run(["--gpus", "2"], RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["value"] is None and "single-GPU" in d["unavailable"]


def test_multi_gpu_launch_ranks():
    r0 = _run(["--gpus", "2"], RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r1 = _run(["--gpus", "2"], RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    assert r0.returncode == 0 and r1.returncode == 0
    assert json.loads(r0.stdout.strip())["unavailable"]
    assert r1.stdout.strip() == ""


def test_reference_arm_rank_other_than_zero_exits_quietly():
    r = _run(["--impl", "reference", "--gpus", "2"], RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    assert r.returncode == 0 and r.stdout.strip() == ""
