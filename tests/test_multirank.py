"""The bench's multi-GPU path is N independent replicas (no collective on the
data path): a barrier, the slowest rank's time and the whole job's units.
Checked here with two gloo ranks on the CPU."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
    rate = bench.replica_rate(15.0, world, slowest * 1e-3)
    q.put((rank, slowest, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_units():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [15.0, 15.0]           # every rank sees the slowest time
    assert all(abs(o[2] - 2 * 15.0 / 15e-3) < 1e-6 for o in out)  # both replicas' units / that time


def test_reference_arm_rank_other_than_zero_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
