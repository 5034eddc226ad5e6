"""bench.py's multi-GPU reading (replicas, one per rank) on the host: the
slowest rank's time counts and the job's throughput adds every rank's tokens.
Two gloo ranks on the CPU stand in for two GPUs (no data-path collective
exists: each rank runs its own copy of the layer)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, device="cpu")
        rate = bench.job_rate(4, env[0], slowest)
        q.put((rank, env, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, slowest, rate in res:
        assert env == (2, rank, rank)
        assert slowest == 15.0
        assert rate == pytest.approx(4 * 2 / 0.015)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, device="cpu") == 3.5
    assert bench.job_rate(8, 1, 2.0) == pytest.approx(4000.0)
