"""The benchmark's multi-rank host logic on two CPU processes (gloo): the
maximum over ranks, the replicas' whole-job rate, and the reference arm's
rank handling.  No GPU is touched."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.rank_env()
        assert (w, r, lr) == (world, rank, rank)
        slowest = bench.max_over_ranks(10.0 + rank, world, "cpu")   # rank 1 is the slower one
        out.put((rank, slowest, bench.job_rate(world, 4.0e9, slowest * 1e-3)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, rate in got:
        assert slowest == 11.0                               # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 4.0e9 / 11.0e-3)    # both ranks' bytes over that time


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
