"""The benchmark's multi-rank plumbing (one process per GPU, independent
replicas of the step): barrier and max-over-ranks timing, checked with two
gloo ranks on the CPU."""

import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), FASA_BENCH_BACKEND="gloo")
    import bench
    r, w, local, pg = bench.dist_setup(world)
    bench.barrier(pg)
    m = bench.max_over_ranks(pg, 10.0 * (rank + 1))
    bench.barrier(pg)
    pg.destroy_process_group()
    q.put((r, w, local, m))


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_world_size_must_match_gpus():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    with pytest.raises(SystemExit):
        bench.dist_setup(2)
