"""Host logic of the multi-GPU bench (replicas): world_size-2 gloo ranks on CPU.

Each replica runs the whole decode pass on its own GPU; the job's time is the
slowest rank's and the job's rate counts every rank's work.  No GPU here: the
aggregation runs on CPU tensors over gloo, and a non-zero rank of the
reference arm exits without work.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, seconds, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(torch, dist, seconds[rank], torch.device("cpu"))
        rate = bench.whole_job_rate(1000, 10, world, t)
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds = [0.25, 0.40]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, rate in got:
        assert t == pytest.approx(0.40)                       # the slowest rank, on every rank
        assert rate == pytest.approx(1000 * 10 * 2 / 0.40)   # both replicas' work over that time


def test_single_process_aggregation_is_identity():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, None, 0.123, None) == 0.123
    assert bench.whole_job_rate(5, 4, 1, 2.0) == pytest.approx(10.0)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
