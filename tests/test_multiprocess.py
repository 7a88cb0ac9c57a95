"""The benchmark's multi-GPU path is replicas only (independent sequences per
GPU, no data-path collective): ranks meet at a barrier around the timed region
and rank 0 reports the maximum time over ranks.  These CPU tests run that
logic with world_size 2 over gloo on 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), PKV_DIST_BACKEND="gloo")
    import bench
    r, w, dist = bench.dist_setup(world)
    assert (r, w) == (rank, world) and dist is not None
    bench.barrier(dist)
    ms = 10.0 * (rank + 1)          # rank 1 is the slowest
    q.put((rank, bench.max_over_ranks(ms, dist)))
    bench.barrier(dist)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_replica_timing_takes_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 20.0, 1: 20.0}


def test_single_process_needs_no_process_group():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_setup(1) == (0, 1, None)
    assert bench.max_over_ranks(3.5, None) == 3.5
