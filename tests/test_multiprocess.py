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


def _shard_worker(rank, world, port, results):
    """One rank of the receiver-sharded convolution (oracle as the compute)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import torch.distributed as dist

    import oracle as O
    import workloads as W
    from clebsch_gordan_tensor_gb300 import shard

    dist.init_process_group("gloo", rank=rank, world_size=world)
    irreps = ("8x0e+8x1o", "0e+1o+2e", "8x0e+8x1o+8x1e+8x2e")
    prob = O.make_problem(*irreps)
    rng = np.random.default_rng(31)
    _, _, gr = W.periodic_cloud(rng, 150)
    x = rng.standard_normal((gr.N, prob.dim1))
    y = rng.standard_normal((gr.E, prob.dim2))
    w = rng.standard_normal((gr.E, prob.wdim))
    g = rng.standard_normal((gr.N, prob.dimo))
    b = shard.receiver_bounds(gr.rowptr, world)
    r0, r1 = int(b[rank]), int(b[rank + 1])
    e0, e1 = int(gr.rowptr[r0]), int(gr.rowptr[r1])
    T = torch.from_numpy

    def conv_fn(rp, snd, xf, ye, we, scale):
        return T(O.conv_forward(prob, rp, snd, xf.numpy(), ye.numpy(), we.numpy(), scale))

    def bwd_fn(rp, snd, xf, ye, we, scale, gf):
        return tuple(T(a) for a in O.conv_backward(prob, rp, snd, xf.numpy(), ye.numpy(),
                                                   we.numpy(), scale, gf.numpy()))

    out = shard.conv_forward(dist, rank, b, gr.rowptr, gr.sender, T(x[r0:r1]), T(y[e0:e1]),
                             T(w[e0:e1]), 0.25, conv_fn)
    gx, gy, gw = shard.conv_backward(dist, rank, b, gr.rowptr, gr.sender, T(x[r0:r1]),
                                     T(y[e0:e1]), T(w[e0:e1]), 0.25, T(g[r0:r1]), bwd_fn)
    results[rank] = (r0, r1, e0, e1, out.numpy(), gx.numpy(), gy.numpy(), gw.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_receiver_sharded_conv_matches_one_rank():
    """Two gloo ranks, each owning a receiver range balanced by edge count:
    forward rows and per-edge gradients equal the one-rank oracle's exactly
    (same edges, same order); grad_x, summed across ranks by the
    reduce-scatter, agrees to rounding."""
    import numpy as np

    import oracle as O
    import workloads as W

    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    irreps = ("8x0e+8x1o", "0e+1o+2e", "8x0e+8x1o+8x1e+8x2e")
    prob = O.make_problem(*irreps)
    rng = np.random.default_rng(31)
    _, _, gr = W.periodic_cloud(rng, 150)
    x = rng.standard_normal((gr.N, prob.dim1))
    y = rng.standard_normal((gr.E, prob.dim2))
    w = rng.standard_normal((gr.E, prob.wdim))
    g = rng.standard_normal((gr.N, prob.dimo))
    out = O.conv_forward(prob, gr.rowptr, gr.sender, x, y, w, 0.25)
    gx, gy, gw = O.conv_backward(prob, gr.rowptr, gr.sender, x, y, w, 0.25, g)
    (a0, a1, ea, eb, *_), (b0, b1, ec, ed, *_) = results[0], results[1]
    assert (a0, a1, b1) == (0, b0, gr.N) and (ea, eb, ed) == (0, ec, gr.E)
    assert abs((eb - ea) - (ed - ec)) <= 2 * int(np.diff(gr.rowptr).max())  # balanced
    for r in range(world):
        r0, r1, e0, e1, o, sx, sy, sw = results[r]
        assert np.array_equal(o, out[r0:r1])
        assert np.array_equal(sy, gy[e0:e1]) and np.array_equal(sw, gw[e0:e1])
        np.testing.assert_allclose(sx, gx[r0:r1], rtol=1e-12, atol=1e-12)


def test_receiver_bounds_balance_edges():
    import numpy as np

    from clebsch_gordan_tensor_gb300 import shard

    rowptr = np.concatenate([[0], np.cumsum(np.random.default_rng(3).integers(0, 60, 1000))])
    for world in (1, 2, 3, 8):
        b = shard.receiver_bounds(rowptr, world)
        assert b[0] == 0 and b[-1] == 1000 and np.all(np.diff(b) >= 0)
        edges = np.diff(rowptr[b])
        assert edges.sum() == rowptr[-1]
        assert edges.max() - edges.min() <= 2 * 60
