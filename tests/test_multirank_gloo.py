"""The benchmark's multi-rank host logic on CPU: two gloo ranks, the way
torchrun launches bench.py with --gpus 2 (independent replicas, max-over-ranks
time, whole-job throughput), plus the reference arm's rank handling."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        own = 1.0 + 0.5 * rank                # rank 1 is the slow one
        times = bench.max_over_ranks(own, "cpu")
        value, t = bench.aggregate(times, 1000.0)
        q.put((r, w, local, times, value, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, (r, w, local, times, value, t) in enumerate(out):
        assert (r, w, local) == (rank, world, rank)
        assert times == [1.5, 1.5]               # max over ranks, seen by both
        assert t == 1.5
        assert value == pytest.approx(2 * 1000.0 / 1.5)   # both replicas' units / slowest time


def test_single_rank_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25, "cpu") == [0.25]
    assert bench.aggregate([0.25], 10.0) == (40.0, 0.25)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
