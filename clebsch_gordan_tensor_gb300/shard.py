"""Receiver-range sharding of the fused convolution across ranks (one GPU per
rank): the partition, each rank's share of the graph, and the two exchanges.

The fused convolution ("An Efficient Sparse Kernel Generator for
O(3)-Equivariant Deep Networks", abstract: the tensor product fused with the
graph convolution around it) partitions by receiver.  Rank r owns a
contiguous receiver range [b_r, b_{r+1}) balanced by edge count (edges are
sorted by receiver), the node rows of that range, and that range's edges.

- Forward: one all-gather of the node features (a rank's edges read senders
  anywhere), then every receiver sums its own edges -- the same edges in the
  same order as on one rank, so its output row is the one-rank row.
- Backward: grad_y and grad_w belong to the rank's edges.  A sender's grad_x
  collects edges held by every rank, so each rank computes its edges'
  contributions for all N nodes and a reduce-scatter (sum over ranks, then
  the rank's rows) hands each rank its node rows.

The tensor-product arithmetic is passed in (the library's fused convolution
on a GPU rank); this module only partitions and exchanges.  Collectives go
through ``torch.distributed`` (NCCL on GPUs, gloo on CPU ranks).
"""
from __future__ import annotations

import numpy as np
import torch


def receiver_bounds(rowptr, world: int) -> np.ndarray:
    """[world + 1] receiver bounds: rank r owns receivers [b[r], b[r+1]), the
    first receiver whose edges start at or after r * E / world opening rank
    r's range (the split the persistent kernels use between CTAs)."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    N, E = rowptr.shape[0] - 1, int(rowptr[-1])
    if world < 1:
        raise ValueError("world must be >= 1")
    targets = [E * r // world for r in range(1, world)]
    inner = np.searchsorted(rowptr[:N], targets, side="left")
    return np.concatenate([[0], np.minimum(inner, N), [N]]).astype(np.int64)


def shard_csr(rowptr, sender, r0: int, r1: int):
    """The rank's share of the receiver-sorted graph: a CSR over all N
    receivers in which only [r0, r1) keep their edges (global node indices),
    its senders, and the edge range [e0, e1) of the full graph it covers."""
    rowptr = np.asarray(rowptr, dtype=np.int64)
    e0, e1 = int(rowptr[r0]), int(rowptr[r1])
    local = np.clip(rowptr - e0, 0, e1 - e0)
    local[: r0 + 1] = 0
    local[r1:] = e1 - e0
    return local.astype(np.int32), np.asarray(sender[e0:e1], dtype=np.int32), e0, e1


def all_gather_rows(dist, local: torch.Tensor, bounds) -> torch.Tensor:
    """Concatenate every rank's node rows (rank r holds rows [b[r], b[r+1]))."""
    world = len(bounds) - 1
    rows = [int(bounds[r + 1] - bounds[r]) for r in range(world)]
    width = local.shape[1:]
    pad = max(rows)
    buf = torch.zeros((pad,) + tuple(width), dtype=local.dtype, device=local.device)
    buf[: local.shape[0]] = local
    parts = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf)
    return torch.cat([p[:n] for p, n in zip(parts, rows)], dim=0)


def reduce_scatter_rows(dist, full: torch.Tensor, bounds, rank: int) -> torch.Tensor:
    """Sum a [N, ...] tensor over ranks and keep this rank's rows."""
    total = full.clone()
    dist.all_reduce(total)
    return total[int(bounds[rank]): int(bounds[rank + 1])]


def conv_forward(dist, rank: int, bounds, rowptr, sender, x_local, y_edges, w_edges, scale,
                 conv_fn):
    """This rank's output rows.  conv_fn(rowptr, sender, x, y, w, scale) is the
    fused convolution over the given CSR (all N nodes, rows outside the rank's
    range empty); y_edges, w_edges hold the rank's edges (per-edge weights) or
    w_edges the shared row."""
    r0, r1 = int(bounds[rank]), int(bounds[rank + 1])
    x_full = all_gather_rows(dist, x_local, bounds)
    rp, snd, _, _ = shard_csr(rowptr, sender, r0, r1)
    out = conv_fn(rp, snd, x_full, y_edges, w_edges, scale)
    return out[r0:r1]


def conv_backward(dist, rank: int, bounds, rowptr, sender, x_local, y_edges, w_edges, scale,
                  grad_out_local, bwd_fn):
    """(grad_x of this rank's node rows, grad_y and grad_w of its edges).
    bwd_fn(rowptr, sender, x, y, w, scale, grad_out) returns the convolution's
    gradient over the given CSR: grad_x [N, ...] with the contributions of its
    edges, grad_y and grad_w per edge."""
    r0, r1 = int(bounds[rank]), int(bounds[rank + 1])
    x_full = all_gather_rows(dist, x_local, bounds)
    rp, snd, _, _ = shard_csr(rowptr, sender, r0, r1)
    N = rp.shape[0] - 1
    g_full = torch.zeros((N,) + tuple(grad_out_local.shape[1:]), dtype=grad_out_local.dtype,
                         device=grad_out_local.device)
    g_full[r0:r1] = grad_out_local
    gx_part, gy, gw = bwd_fn(rp, snd, x_full, y_edges, w_edges, scale, g_full)
    return reduce_scatter_rows(dist, gx_part, bounds, rank), gy, gw
