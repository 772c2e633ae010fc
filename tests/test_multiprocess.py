"""Multi-process (N > 1) host logic of the benchmark, on CPU with gloo.

Every rank runs an independent replica of the workload (there is no exchange
on the data path); the job time is the slowest rank's, taken with one
all-reduce(MAX).  Run as two spawned processes on 127.0.0.1.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist, r, ws = bench.dist_setup()
    assert (r, ws) == (rank, world) and dist is not None
    # each rank "timed" a different duration; all must agree on the max
    results[rank] = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_timing():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 15.0, 1: 15.0}


def test_single_process_has_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench

    dist, rank, world = bench.dist_setup()
    assert dist is None and (rank, world) == (0, 1)
    assert bench.max_over_ranks(None, 3.5) == 3.5
