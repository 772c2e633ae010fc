"""Seeded synthetic inputs for the Clebsch-Gordan tensor-product workloads.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds none of the library's arithmetic (tensor product, spherical harmonics,
CG coefficients, the radial network): it draws random numbers and builds
neighbour graphs, all in numpy.  Conv workloads carry the radial network's
parameters; the per-edge weights are computed from them by the library on the
GPU and by the oracle on the host.

The pages measure on QM9, MACE foundation-model inference and water MD (see
"An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks",
abstract; NVIDIA SE(3)-Transformer blog, Fig. 2-3; "Speeding Up MACE",
abstract).  None of those datasets is used; these recipes stand in for them
with the same shapes: MACE-like node features of l <= 2 and edge spherical
harmonics of l <= 3 on a dense periodic atom cloud, and small fully connected
molecules for the TFN-style layer.

Every generator takes a seed for ``numpy.random.default_rng`` and draws in the
order written in its docstring.  fp32 workloads draw float32 normals directly
(``standard_normal(dtype=float32)``); fp64 workloads draw float64.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Irreps (in1, in2, out) of the five workloads.
IRREPS_TP16 = ("16x0e+16x1o", "0e+1o+2e", "16x0e+16x1o+16x2e")
IRREPS_MACE128 = ("128x0e+128x1o+128x2e", "0e+1o+2e+3o",
        "128x0e+128x1o+128x1e+128x2o+128x2e+128x3o+128x3e")
IRREPS_CONV64 = ("64x0e+64x1o+64x2e", "0e+1o+2e+3o", "64x0e+64x1o+64x1e+64x2o+64x2e+64x3o+64x3e")
IRREPS_CONV128 = ("128x0e+128x1o+128x2e", "0e+1o+2e+3o",
        "128x0e+128x1o+128x1e+128x2o+128x2e+128x3o+128x3e")
IRREPS_TFN32 = ("32x0e+32x1o+32x2e+32x3o", "0e+1o+2e+3o", "32x0e+32x1o+32x2e+32x3o")
# the small-molecule TFN layer with keys and values from one TFN: channels doubled
IRREPS_TFN_KV64 = ("64x0e+64x1o+64x2e+64x3o", "0e+1o+2e+3o", "64x0e+64x1o+64x2e+64x3o")


def irreps_dim(s: str) -> int:
    d = 0
    for tok in s.split("+"):
        mul, rest = tok.split("x") if "x" in tok else ("1", tok)
        d += int(mul) * (2 * int(rest[:-1]) + 1)
    return d


def normal(rng, shape, dtype):
    if np.dtype(dtype) == np.float32:
        return rng.standard_normal(shape, dtype=np.float32)
    return rng.standard_normal(shape).astype(dtype, copy=False)


@dataclass
class Graph:
    """Receiver-sorted CSR plus the sender-grouped view used by gradients.

    rowptr[N+1], sender[E]: edges e in rowptr[n]..rowptr[n+1]-1 have receiver n,
    sorted by (receiver, sender).  s_rowptr[N+1], s_perm[E], s_recv[E]: the
    edges grouped by sender s are s_perm[s_rowptr[s]..s_rowptr[s+1]-1] (in
    increasing edge index), and s_recv[j] = receiver of edge s_perm[j].
    vec[E, 3] = pos[receiver] - pos[sender] (minimum image when periodic)."""
    N: int
    rowptr: np.ndarray
    sender: np.ndarray
    receiver: np.ndarray
    vec: np.ndarray
    s_rowptr: np.ndarray
    s_perm: np.ndarray
    s_recv: np.ndarray

    @property
    def E(self) -> int:
        return int(self.sender.shape[0])


def make_graph(N: int, receiver: np.ndarray, sender: np.ndarray, vec: np.ndarray) -> Graph:
    """Sort edges by (receiver, sender) and build both CSR views."""
    receiver = np.asarray(receiver, dtype=np.int64)
    sender = np.asarray(sender, dtype=np.int64)
    order = np.lexsort((sender, receiver))
    receiver, sender, vec = receiver[order], sender[order], np.asarray(vec)[order]
    rowptr = np.zeros(N + 1, dtype=np.int64)
    np.cumsum(np.bincount(receiver, minlength=N), out=rowptr[1:])
    s_order = np.argsort(sender, kind="stable")
    s_rowptr = np.zeros(N + 1, dtype=np.int64)
    np.cumsum(np.bincount(sender, minlength=N), out=s_rowptr[1:])
    return Graph(N, rowptr.astype(np.int32), sender.astype(np.int32),
                 receiver.astype(np.int32), vec, s_rowptr.astype(np.int32),
                 s_order.astype(np.int32), receiver[s_order].astype(np.int32))


def periodic_cloud(rng, N: int, density: float = 0.1, cutoff: float = 5.0):
    """N atoms uniform in a periodic cube of side (N/density)^(1/3); directed
    edges for every ordered pair closer than ``cutoff`` (strict, minimum image),
    no self edges.  Draws: positions [N, 3] uniform in [0, L)."""
    from scipy.spatial import cKDTree

    L = (N / density) ** (1.0 / 3.0)
    if L <= 2 * cutoff:
        raise ValueError("box too small for the minimum-image convention")
    pos = rng.uniform(0.0, L, size=(N, 3))
    tree = cKDTree(pos, boxsize=L)
    pairs = tree.query_pairs(cutoff, output_type="ndarray")
    i, j = pairs[:, 0], pairs[:, 1]
    recv = np.concatenate([i, j])
    send = np.concatenate([j, i])
    d = pos[recv] - pos[send]
    d -= L * np.round(d / L)
    keep = np.einsum("ij,ij->i", d, d) < cutoff * cutoff
    return pos, L, make_graph(N, recv[keep], send[keep], d[keep])


def molecules(rng, n_mol: int, n_min: int = 9, n_max: int = 29, step=(1.0, 1.6)):
    """n_mol molecules of U{n_min..n_max} atoms placed by a random walk with
    step lengths U(step) along uniform random directions; every ordered pair of
    distinct atoms inside one molecule is an edge.
    Draws: sizes [n_mol]; then per molecule, step lengths [n-1] and step
    directions [n-1, 3] (normal, normalised)."""
    sizes = rng.integers(n_min, n_max + 1, size=n_mol)
    pos_list, recv, send = [], [], []
    base = 0
    for n in sizes:
        n = int(n)
        lengths = rng.uniform(step[0], step[1], size=n - 1)
        dirs = rng.standard_normal((n - 1, 3))
        dirs /= np.linalg.norm(dirs, axis=1, keepdims=True)
        p = np.zeros((n, 3))
        p[1:] = np.cumsum(dirs * lengths[:, None], axis=0)
        pos_list.append(p)
        a, b = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        m = a != b
        recv.append(a[m] + base)
        send.append(b[m] + base)
        base += n
    pos = np.concatenate(pos_list)
    recv, send = np.concatenate(recv), np.concatenate(send)
    return pos, make_graph(base, recv, send, pos[recv] - pos[send])


def radial_params(rng, n_out: int, n_basis: int = 8, hidden: int = 64, dtype=np.float32):
    """Parameters of the fixed random radial network that produces the per-edge
    weights (Bessel(n_basis) -> Linear(n_basis, hidden) -> SiLU ->
    Linear(hidden, n_out), no biases): W1 [n_basis, hidden] ~ N(0,1)/sqrt(n_basis)
    and W2 [hidden, n_out] ~ N(0,1)/sqrt(hidden), both rounded to the workload
    dtype.  Draws: W1, then W2 (float64 normals)."""
    W1 = rng.standard_normal((n_basis, hidden)) / np.sqrt(n_basis)
    W2 = rng.standard_normal((hidden, n_out)) / np.sqrt(hidden)
    return W1.astype(dtype), W2.astype(dtype)


# -------------------------------------------------------------- workloads --

def standalone(seed: int, irreps, B: int, wdim: int, w_scale: float = 1.0,
               dtype=np.float32) -> dict:
    """Standalone tensor-product inputs.  Draws, in order: x [B, dim1] ~ N(0,1);
    v [B, 3] ~ N(0,1) (the second operand is the SH of v); w [B, wdim] ~ N(0,1)
    times w_scale."""
    rng = np.random.default_rng(seed)
    x = normal(rng, (B, irreps_dim(irreps[0])), dtype)
    v = normal(rng, (B, 3), dtype)
    w = normal(rng, (B, wdim), dtype)
    if w_scale != 1.0:
        w *= np.asarray(w_scale, dtype=dtype)
    return dict(irreps=irreps, B=B, x=x, vec=v, w=w, lmax=_lmax(irreps[1]),
                dtype=np.dtype(dtype))


def _lmax(irreps_in2: str) -> int:
    return max(int(t.split("x")[-1][:-1]) for t in irreps_in2.split("+"))


def tp16_b1000(B: int = 1000) -> dict:
    """Standalone TP, fp32, B = 1000, 16x0e+16x1o (x) SH(l<=2) -> 16x(0e,1o,2e),
    7 paths, per-sample weights N(0,1), seed 0."""
    return standalone(0, IRREPS_TP16, B, wdim=7 * 16, dtype=np.float32)


def mace128_b200k(B: int = 200_000) -> dict:
    """MACE-like standalone TP, fp32, B = 200,000, 128x(0e,1o,2e) (x) SH(l<=3)
    -> 128x(0e,1o,1e,2o,2e,3o,3e), 24 paths, weights N(0,1)/sqrt(24), seed 1."""
    return standalone(1, IRREPS_MACE128, B, wdim=24 * 128, w_scale=1.0 / np.sqrt(24.0), dtype=np.float32)


def mace128_uvw_b200k(B: int = 200_000) -> dict:
    """The 200,000-sample, 128-channel standalone inputs (x, v from seed 1, as
    ``mace128_b200k`` draws them) under a 'uvw' product: one [128, 128] matrix per
    path shared by all samples, W ~ N(0,1)/sqrt(128) from seed 101 (24 paths,
    path-major, row-major)."""
    cfg = mace128_b200k(B)
    cfg.pop("w")
    rng = np.random.default_rng(101)
    cfg["W"] = normal(rng, (24 * 128 * 128,), np.float32) * np.float32(1.0 / np.sqrt(128.0))
    return cfg


def conv_cloud(seed: int, irreps, N: int, n_paths: int, dtype) -> dict:
    """Fused graph convolution on a periodic atom cloud (density 0.1 / A^3,
    cutoff 5 A).  Draws, in order: positions (``periodic_cloud``); x [N, dim1]
    ~ N(0,1); radial network parameters (``radial_params``, n_out = n_paths *
    mul).  The per-edge weights are that network applied to the edge lengths;
    this module does not evaluate it (the library and the oracle each do).
    scale = 1 / average degree = N / E."""
    rng = np.random.default_rng(seed)
    pos, L, g = periodic_cloud(rng, N)
    mul = int(irreps[0].split("x")[0])
    x = normal(rng, (N, irreps_dim(irreps[0])), dtype)
    W1, W2 = radial_params(rng, n_paths * mul, dtype=dtype)
    return dict(irreps=irreps, graph=g, pos=pos, box=L, x=x, vec=g.vec.astype(dtype), W1=W1,
                W2=W2, cutoff=5.0, lmax=3, scale=float(N) / float(max(g.E, 1)),
                dtype=np.dtype(dtype))


def tfn_kv64_mol1000(n_mol: int = 1000) -> dict:
    """The TFN workload's 1000 molecules (same seed, same graph) with 64 channels per
    irrep: the keys and values of an SE(3)-Transformer attention layer from one
    TFN with doubled channels instead of two.  Draws, in order: molecules; x
    [N, 1024] ~ N(0,1); w [E, 23 * 64] ~ N(0,1)/sqrt(23); g [N, 1024] ~ N(0,1)
    (output cotangent)."""
    rng = np.random.default_rng(4)
    pos, g = molecules(rng, n_mol)
    x = normal(rng, (g.N, 1024), np.float32)
    w = normal(rng, (g.E, 23 * 64), np.float32) * np.float32(1.0 / np.sqrt(23.0))
    go = normal(rng, (g.N, 1024), np.float32)
    return dict(irreps=IRREPS_TFN_KV64, graph=g, pos=pos, x=x, vec=g.vec.astype(np.float32), w=w, g=go,
                lmax=3, scale=1.0, dtype=np.dtype(np.float32))


def conv64_cloud10k(N: int = 10_000) -> dict:
    """Fused conv, fp32, N = 10,000 atoms, 64x(0e,1o,2e) (x) SH(l<=3) -> 64 x 7
    irreps, 24 paths, radial-MLP weights, seed 2."""
    return conv_cloud(2, IRREPS_CONV64, N, 24, np.float32)


def conv128_f64_cloud5k(N: int = 5_000) -> dict:
    """Fused conv, fp64, N = 5,000 atoms, 128 channels, seed 3, forward only."""
    return conv_cloud(3, IRREPS_CONV128, N, 24, np.float64)


def tfn32_mol1000(n_mol: int = 1000) -> dict:
    """TFN-style layer on small molecules, fp32, seed 4.  Draws, in order:
    molecules (``molecules``); x [N, 512] ~ N(0,1); w [E, 736] ~ N(0,1)/sqrt(23);
    c [N, 512] ~ N(0,1) (energy E = sum c * out); gF [N, 3] ~ N(0,1) (force
    cotangent, L = sum gF * F).  No 1/degree scale."""
    rng = np.random.default_rng(4)
    pos, g = molecules(rng, n_mol)
    x = normal(rng, (g.N, 512), np.float32)
    w = normal(rng, (g.E, 23 * 32), np.float32) * np.float32(1.0 / np.sqrt(23.0))
    c = normal(rng, (g.N, 512), np.float32)
    gF = normal(rng, (g.N, 3), np.float32)
    return dict(irreps=IRREPS_TFN32, graph=g, pos=pos, x=x, vec=g.vec.astype(np.float32), w=w, c=c,
                gF=gF, lmax=3, scale=1.0, dtype=np.dtype(np.float32))
