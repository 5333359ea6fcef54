"""The benchmark's multi-process host logic on CPU with the gloo backend:
each rank runs an independent replica (the path has no exchange step), the
slowest rank's time is taken, and the whole-job throughput counts the units
of every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        seconds = 1.0 + r  # rank r "took" 1 + r seconds
        slowest = bench.reduce_max(seconds, w)
        value = bench.whole_job_value(100.0, slowest, w)
        q.put((r, w, slowest, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank_and_count_all_units(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, w, slowest, value in res:
        assert w == world
        assert slowest == pytest.approx(float(world))      # max over ranks of 1 + r
        assert value == pytest.approx(100.0 * world / world)  # all ranks' units / slowest time


def test_single_process_defaults():
    os.environ.pop("WORLD_SIZE", None)
    w, r, l = bench.dist_env()
    assert (w, r, l) == (1, 0, 0)
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.whole_job_value(10.0, 2.0, 1) == 5.0
