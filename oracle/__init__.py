"""Oracle for the Clebsch-Gordan tensor product -- TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 CPU restatement of what the GPU library computes, used to
check it.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package; the product path
(``clebsch_gordan_tensor_gb300``) never does and shares no code with it.

The arithmetic lives in ``cgtp_oracle.c`` (compiled with gcc on first use).
This module adds what is plain bookkeeping: parsing irreps strings, listing the
'uvu' paths, and the double-backward identity written as sums of the
first-order pieces.

Sources: "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
Networks" (arXiv 2501.13986), abstract -- the CG tensor product of two dense
irrep vectors with a structured sparse tensor, fused with a graph convolution,
with its gradient and the higher partial derivatives used for forces; NVIDIA's
SE(3)-Transformer blog, section "TFN fusion" -- degree-d features have
dimension 2d+1 and pairwise degree convolutions are summed per output degree.

Parity pins: every function here is pinned in ``tests/test_oracle_*.py`` against
textbook closed forms, library routines (sympy CG, scipy spherical harmonics),
invariants (orthogonality, equivariance under rotations and inversion, adjoint
identities) or finite differences.  The pages print no worked numbers, so the
absolute values are "parity unpinned" against the pages themselves.
"""
from __future__ import annotations

import ctypes
import os
import re
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libcgtp_oracle.so")
_SRC = os.path.join(_HERE, "cgtp_oracle.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared",
                               "-ffp-contract=off", _SRC, "-lm", "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


class _Path(ctypes.Structure):
    _fields_ = [("l1", ctypes.c_int), ("l2", ctypes.c_int), ("l3", ctypes.c_int),
                ("mul", ctypes.c_int), ("off1", ctypes.c_int64), ("off2", ctypes.c_int64),
                ("off3", ctypes.c_int64), ("offw", ctypes.c_int64)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            d, i64, i32 = ctypes.c_double, ctypes.c_int64, ctypes.c_int
            pd = P(d)
            pi32 = P(ctypes.c_int32)
            lib.oracle_cg_real.argtypes = [i32, i32, i32, pd]
            lib.oracle_cg_complex.argtypes = [i32] * 6
            lib.oracle_cg_complex.restype = d
            lib.oracle_sh.argtypes = [i32, i64, pd, pd]
            lib.oracle_sh_vjp.argtypes = [i32, i64, pd, pd, pd]
            lib.oracle_sh_jvp.argtypes = [i32, i64, pd, pd, pd]
            lib.oracle_sh_hvp.argtypes = [i32, i64, pd, pd, pd, pd]
            lib.oracle_tp_forward.argtypes = [i32, P(_Path), i64, i64, i64, i64, i64, i64,
                                              pd, pd, pd, pd]
            lib.oracle_tp_backward.argtypes = [i32, P(_Path), i64, i64, i64, i64, i64, i64,
                                               pd, pd, pd, pd, pd, pd, pd]
            lib.oracle_conv_forward.argtypes = [i32, P(_Path), i64, i64, pi32, pi32, i64, i64,
                                                i64, i64, i64, pd, pd, pd, d, pd, i64,
                                                P(ctypes.c_int64)]
            lib.oracle_conv_backward.argtypes = [i32, P(_Path), i64, i64, pi32, pi32, i64, i64,
                                                 i64, i64, i64, pd, pd, pd, d, pd, pd, pd, pd,
                                                 P(ctypes.c_uint8), P(ctypes.c_uint8)]
            lib.oracle_edge_forces.argtypes = [i64, i64, pi32, pi32, pd, pd]
            for f in ("oracle_cg_real", "oracle_sh", "oracle_sh_vjp", "oracle_sh_jvp", "oracle_sh_hvp",
                      "oracle_tp_forward", "oracle_tp_backward", "oracle_conv_forward",
                      "oracle_conv_backward", "oracle_edge_forces"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a, t=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(t))


# --------------------------------------------------------------- irreps ---

_IRREP = re.compile(r"^\s*(?:(\d+)\s*x\s*)?(\d+)\s*([eo])\s*$")


def parse_irreps(s: str):
    """'16x0e+16x1o' -> [(mul, l, parity)] with parity +1 (e) / -1 (o)."""
    out = []
    for tok in s.split("+"):
        m = _IRREP.match(tok)
        if not m:
            raise ValueError(f"bad irrep {tok!r} in {s!r}")
        mul = int(m.group(1)) if m.group(1) else 1
        out.append((mul, int(m.group(2)), 1 if m.group(3) == "e" else -1))
    return out


def irreps_dim(irreps) -> int:
    return sum(mul * (2 * l + 1) for mul, l, _ in irreps)


@dataclass
class Problem:
    """Irreps of the two inputs and the output plus the 'uvu' path list."""
    in1: list
    in2: list
    out: list
    paths: list  # (i1, i2, i3, l1, l2, l3, mul, off1, off2, off3, offw)
    dim1: int
    dim2: int
    dimo: int
    wdim: int

    def ctypes_paths(self):
        arr = (_Path * max(1, len(self.paths)))()
        for k, (_, _, _, l1, l2, l3, mul, o1, o2, o3, ow) in enumerate(self.paths):
            arr[k] = _Path(l1, l2, l3, mul, o1, o2, o3, ow)
        return arr


def make_problem(irreps_in1: str, irreps_in2: str, irreps_out: str) -> Problem:
    """All parity-allowed 'uvu' paths: for every (in1, in2, out) irrep triple with
    |l1-l2| <= l3 <= l1+l2, p3 = p1 p2, mul(out) = mul(in1), mul(in2) = 1.
    Paths are listed with in1 outermost, then in2, then out; weights of one
    path form one block of mul in that order."""
    a, b, c = parse_irreps(irreps_in1), parse_irreps(irreps_in2), parse_irreps(irreps_out)

    def offsets(ir):
        off, res = 0, []
        for mul, l, _ in ir:
            res.append(off)
            off += mul * (2 * l + 1)
        return res

    oa, ob, oc = offsets(a), offsets(b), offsets(c)
    paths, offw = [], 0
    for i1, (m1, l1, p1) in enumerate(a):
        for i2, (m2, l2, p2) in enumerate(b):
            for i3, (m3, l3, p3) in enumerate(c):
                if abs(l1 - l2) <= l3 <= l1 + l2 and p3 == p1 * p2 and m3 == m1 and m2 == 1:
                    paths.append((i1, i2, i3, l1, l2, l3, m1, oa[i1], ob[i2], oc[i3], offw))
                    offw += m1
    return Problem(a, b, c, paths, irreps_dim(a), irreps_dim(b), irreps_dim(c), offw)


# ------------------------------------------------------------------- CG ---

def cg_complex(l1: int, m1: int, l2: int, m2: int, l3: int, m3: int) -> float:
    """<l1 m1 l2 m2 | l3 m3> (Condon-Shortley phase), Racah's closed form."""
    return float(_load().oracle_cg_complex(l1, m1, l2, m2, l3, m3))


def cg_real(l1: int, l2: int, l3: int) -> np.ndarray:
    """Real-basis CG tensor [2l1+1, 2l2+1, 2l3+1] (zero if the triangle rule fails)."""
    out = np.zeros((2 * l1 + 1) * (2 * l2 + 1) * (2 * l3 + 1))
    r = _load().oracle_cg_real(l1, l2, l3, _p(out))
    if r < 0:
        raise ValueError("l out of range")
    return out.reshape(2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1)


# ------------------------------------------------- spherical harmonics ---

def sh(lmax: int, vec) -> np.ndarray:
    v = _f64(vec).reshape(-1, 3)
    y = np.empty((v.shape[0], (lmax + 1) ** 2))
    if _load().oracle_sh(lmax, v.shape[0], _p(v), _p(y)):
        raise ValueError("lmax out of range")
    return y


def sh_vjp(lmax: int, vec, grad_y) -> np.ndarray:
    v, g = _f64(vec).reshape(-1, 3), _f64(grad_y)
    out = np.empty_like(v)
    _load().oracle_sh_vjp(lmax, v.shape[0], _p(v), _p(g), _p(out))
    return out


def sh_jvp(lmax: int, vec, tangent_vec) -> np.ndarray:
    v, t = _f64(vec).reshape(-1, 3), _f64(tangent_vec).reshape(-1, 3)
    out = np.empty((v.shape[0], (lmax + 1) ** 2))
    _load().oracle_sh_jvp(lmax, v.shape[0], _p(v), _p(t), _p(out))
    return out


def sh_hvp(lmax: int, vec, grad_y, tangent_vec) -> np.ndarray:
    """Second derivative of grad_y . Y(vec) in vec, applied to tangent_vec:
    the derivative of ``sh_vjp`` along tangent_vec with grad_y held fixed."""
    v, g = _f64(vec).reshape(-1, 3), _f64(grad_y)
    t = _f64(tangent_vec).reshape(-1, 3)
    out = np.empty_like(v)
    _load().oracle_sh_hvp(lmax, v.shape[0], _p(v), _p(g), _p(t), _p(out))
    return out


# --------------------------------------------------------- tensor product --

def _wstride(prob, w, rows):
    w = _f64(w)
    if w.ndim == 1:
        return w, 0
    return w, prob.wdim


def tp_forward(prob: Problem, x, y, w) -> np.ndarray:
    """out[b] = sum over paths of the 'uvu' CG product of x[b], y[b], w[b]
    (a 1-D ``w`` is one weight row shared by every sample)."""
    x, y = _f64(x), _f64(y)
    B = x.shape[0]
    w, ws = _wstride(prob, w, B)
    out = np.zeros((B, prob.dimo))
    r = _load().oracle_tp_forward(len(prob.paths), prob.ctypes_paths(), B, prob.dim1,
                                  prob.dim2, prob.wdim, prob.dimo, ws, _p(x), _p(y), _p(w),
                                  _p(out))
    assert r == 0
    return out


def tp_backward(prob: Problem, x, y, w, g):
    """(dL/dx, dL/dy, dL/dw) for dL/dout = g."""
    x, y, g = _f64(x), _f64(y), _f64(g)
    B = x.shape[0]
    w, ws = _wstride(prob, w, B)
    gx, gy = np.zeros_like(x), np.zeros_like(y)
    gw = np.zeros((B, prob.wdim)) if ws else np.zeros(prob.wdim)
    r = _load().oracle_tp_backward(len(prob.paths), prob.ctypes_paths(), B, prob.dim1,
                                   prob.dim2, prob.wdim, prob.dimo, ws, _p(x), _p(y), _p(w),
                                   _p(g), _p(gx), _p(gy), _p(gw))
    assert r == 0
    return gx, gy, gw


def tp_double_backward(prob: Problem, x, y, w, g, ggx=None, ggy=None, ggw=None):
    """Gradients of S = <ggx, dL/dx> + <ggy, dL/dy> + <ggw, dL/dw> with respect
    to x, y, w and g, where (dL/dx, dL/dy, dL/dw) = tp_backward(x, y, w, g).

    The pages name "a novel identity for the higher partial derivatives" but do
    not state it.  Reading: f(x, y, w) is linear in each argument, so with the
    first-order partials f_x, f_y, f_w,
      d_g = f(ggx, y, w) + f(x, ggy, w) + f(x, y, ggw)
      d_x = f_x(g; ggy, w) + f_x(g; y, ggw)
      d_y = f_y(g; ggx, w) + f_y(g; x, ggw)
      d_w = f_w(g; ggx, y) + f_w(g; x, ggy)
    Absent cotangents are zero.  Returns (d_x, d_y, d_w, d_g)."""
    x, y, w, g = _f64(x), _f64(y), _f64(w), _f64(g)
    z = lambda a: np.zeros_like(a)
    ggx = z(x) if ggx is None else _f64(ggx)
    ggy = z(y) if ggy is None else _f64(ggy)
    ggw = z(w) if ggw is None else _f64(ggw)
    d_g = tp_forward(prob, ggx, y, w) + tp_forward(prob, x, ggy, w) + tp_forward(prob, x, y, ggw)
    a = tp_backward(prob, x, ggy, w, g)   # f_x(g; ggy, w), f_w(g; x, ggy)
    b = tp_backward(prob, x, y, ggw, g)   # f_x(g; y, ggw), f_y(g; x, ggw)
    c = tp_backward(prob, ggx, y, w, g)   # f_y(g; ggx, w), f_w(g; ggx, y)
    return a[0] + b[0], c[1] + b[1], c[2] + a[2], d_g


# ------------------------------------------------------ graph convolution --

def _check_graph(prob, rowptr, sender, x, y, w, ws):
    N, E = rowptr.shape[0] - 1, sender.shape[0]
    if x.shape != (N, prob.dim1):
        raise ValueError(f"x has shape {x.shape}, expected {(N, prob.dim1)}")
    if y.shape != (E, prob.dim2):
        raise ValueError(f"y has shape {y.shape}, expected {(E, prob.dim2)}")
    if ws and w.shape != (E, prob.wdim):
        raise ValueError(f"w has shape {w.shape}, expected {(E, prob.wdim)}")
    if rowptr[0] != 0 or rowptr[-1] != E or np.any(np.diff(rowptr) < 0):
        raise ValueError("rowptr is not a CSR row pointer over the edges")
    if E and (sender.min() < 0 or sender.max() >= N):
        raise ValueError("sender index out of range")


def conv_forward(prob: Problem, rowptr, sender, x, y, w, scale: float, receivers=None):
    """out[n] = scale * sum over the receiver's edges, in edge order, of
    TP(x[sender[e]], y[e], w[e]).  With ``receivers`` only those rows are
    computed (the others stay zero)."""
    rowptr, sender = _i32(rowptr), _i32(sender)
    x, y = _f64(x), _f64(y)
    N, E = rowptr.shape[0] - 1, sender.shape[0]
    w, ws = _wstride(prob, w, E)
    _check_graph(prob, rowptr, sender, x, y, w, ws)
    out = np.zeros((N, prob.dimo))
    sel = None if receivers is None else np.ascontiguousarray(receivers, dtype=np.int64)
    r = _load().oracle_conv_forward(
        len(prob.paths), prob.ctypes_paths(), N, E, _p(rowptr, ctypes.c_int32),
        _p(sender, ctypes.c_int32), prob.dim1, prob.dim2, prob.wdim, prob.dimo, ws, _p(x),
        _p(y), _p(w), float(scale), _p(out), 0 if sel is None else sel.shape[0],
        _p(sel, ctypes.c_int64))
    assert r == 0
    return out


def conv_backward(prob: Problem, rowptr, sender, x, y, w, scale: float, g, nodes=None,
                  edges=None):
    """(dL/dx [N, dim1], dL/dy [E, dim2], dL/dw [E, wdim]) for dL/dout = g.
    dL/dx[s] sums over the edges whose sender is s, in edge order.  ``nodes`` /
    ``edges`` restrict which rows are computed (others stay zero)."""
    rowptr, sender = _i32(rowptr), _i32(sender)
    x, y, g = _f64(x), _f64(y), _f64(g)
    N, E = rowptr.shape[0] - 1, sender.shape[0]
    w, ws = _wstride(prob, w, E)
    _check_graph(prob, rowptr, sender, x, y, w, ws)
    g = g.reshape(N, prob.dimo)
    gx, gy = np.zeros((N, prob.dim1)), np.zeros((E, prob.dim2))
    gw = np.zeros((E, prob.wdim)) if ws else np.zeros(prob.wdim)
    nm = em = None
    if nodes is not None:
        nm = np.zeros(N, dtype=np.uint8)
        nm[np.asarray(nodes)] = 1
    if edges is not None:
        em = np.zeros(E, dtype=np.uint8)
        em[np.asarray(edges)] = 1
    r = _load().oracle_conv_backward(
        len(prob.paths), prob.ctypes_paths(), N, E, _p(rowptr, ctypes.c_int32),
        _p(sender, ctypes.c_int32), prob.dim1, prob.dim2, prob.wdim, prob.dimo, ws, _p(x),
        _p(y), _p(w), float(scale), _p(g), _p(gx), _p(gy), _p(gw), _p(nm, ctypes.c_uint8),
        _p(em, ctypes.c_uint8))
    assert r == 0
    return gx, gy, gw


def conv_double_backward(prob: Problem, rowptr, sender, x, y, w, scale, g, ggx=None, ggy=None,
                         ggw=None):
    """The trilinear identity of ``tp_double_backward`` applied to the fused
    convolution (gather by sender, TP per edge, receiver sum, scale).
    Returns (d_x, d_y, d_w, d_g)."""
    x, y, w, g = _f64(x), _f64(y), _f64(w), _f64(g)
    z = lambda a: np.zeros_like(a)
    ggx = z(x) if ggx is None else _f64(ggx)
    ggy = z(y) if ggy is None else _f64(ggy)
    ggw = z(w) if ggw is None else _f64(ggw)
    f = lambda a, b, c: conv_forward(prob, rowptr, sender, a, b, c, scale)
    bwd = lambda a, b, c: conv_backward(prob, rowptr, sender, a, b, c, scale, g)
    d_g = f(ggx, y, w) + f(x, ggy, w) + f(x, y, ggw)
    a = bwd(x, ggy, w)
    b = bwd(x, y, ggw)
    c = bwd(ggx, y, w)
    return a[0] + b[0], c[1] + b[1], c[2] + a[2], d_g


def edge_forces(rowptr, sender, dEdr) -> np.ndarray:
    """F_i = -sum_e dE/dr_e (delta(i, recv e) - delta(i, send e)),
    r_e = pos[recv] - pos[send]."""
    rowptr, sender = _i32(rowptr), _i32(sender)
    d = _f64(dEdr).reshape(-1, 3)
    N = rowptr.shape[0] - 1
    if d.shape[0] != sender.shape[0] or (sender.size and (sender.min() < 0 or sender.max() >= N)):
        raise ValueError("dEdr / sender do not match the graph")
    F = np.zeros((N, 3))
    _load().oracle_edge_forces(N, sender.shape[0], _p(rowptr, ctypes.c_int32),
                               _p(sender, ctypes.c_int32), _p(d), _p(F))
    return F


# ------------------------------------------------------ radial network ---
#
# NVIDIA's SE(3)-Transformer blog, section "Fused key and value computation":
# the radial profile inside a TFN layer is a fully connected network of the
# edge length, and it supplies the per-edge weights of the tensor product.
# The benchmark workload fixes its shape: 8 Bessel functions of the edge
# length -> Linear(8, hidden) -> SiLU -> Linear(hidden, paths * mul), no
# biases, no envelope.  Written here in fp64 with numpy matmuls as the only
# library steps.

def radial_basis(r, n_basis: int, cutoff: float) -> np.ndarray:
    """b_n(r) = sqrt(2/rc) sin(n pi r / rc) / r for n = 1..n_basis, with its
    limit sqrt(2/rc) n pi / rc at r = 0.  Returns [E, n_basis]."""
    r = _f64(r).reshape(-1, 1)
    n = np.arange(1, n_basis + 1, dtype=np.float64).reshape(1, -1)
    k = n * np.pi / cutoff
    safe = np.where(r > 0.0, r, 1.0)
    b = np.sin(k * r) / safe
    b = np.where(r > 0.0, b, k)
    return np.sqrt(2.0 / cutoff) * b


def silu(a):
    """a * sigmoid(a)."""
    return a / (1.0 + np.exp(-a))


def radial_forward(vec, W1, W2, cutoff: float = 5.0, out_dtype=np.float64,
                   chunk: int = 1 << 15):
    """Per-edge weights of the radial network.  vec [E, 3] (edge vectors; only
    their length is used), W1 [n_basis, hidden], W2 [hidden, n_out].
    Returns (w [E, n_out] in out_dtype, h [E, hidden] fp64): h is the hidden
    activation silu(basis @ W1), w = h @ W2.  Rows are done in chunks of
    ``chunk`` edges so large workloads fit in host memory."""
    v = np.asarray(vec).reshape(-1, 3)
    W1, W2 = _f64(W1), _f64(W2)
    if W1.ndim != 2 or W2.ndim != 2 or W1.shape[1] != W2.shape[0]:
        raise ValueError("W1 [n_basis, hidden] and W2 [hidden, n_out] do not match")
    E = v.shape[0]
    w = np.empty((E, W2.shape[1]), dtype=out_dtype)
    h = np.empty((E, W1.shape[1]))
    for a in range(0, E, chunk):
        r = np.linalg.norm(_f64(v[a:a + chunk]), axis=1)
        h[a:a + chunk] = silu(radial_basis(r, W1.shape[0], cutoff) @ W1)
        w[a:a + chunk] = h[a:a + chunk] @ W2
    return w, h


def radial_backward(vec, W1, W2, grad_w, cutoff: float = 5.0):
    """Vector-Jacobian product of ``radial_forward``'s w: returns
    (grad_vec [E, 3], grad_W1, grad_W2) for the cotangent grad_w [E, n_out].
    Chain: gh = grad_w W2^T; gpre = gh * silu'(pre) with
    silu'(a) = s (1 + a (1 - s)), s = sigmoid(a); gW2 = h^T grad_w;
    gW1 = b^T gpre; gb = gpre W1^T; dr = sum_n gb_n db_n/dr with
    db_n/dr = sqrt(2/rc) (k_n cos(k_n r) / r - sin(k_n r) / r^2); grad_vec =
    dr vec / r (zero at r = 0, where the basis is flat)."""
    v = _f64(vec).reshape(-1, 3)
    W1, W2, g = _f64(W1), _f64(W2), _f64(grad_w)
    r = np.linalg.norm(v, axis=1)
    b = radial_basis(r, W1.shape[0], cutoff)
    pre = b @ W1
    s = 1.0 / (1.0 + np.exp(-pre))
    h = pre * s
    gh = g @ W2.T
    gpre = gh * s * (1.0 + pre * (1.0 - s))
    gW2 = h.T @ g
    gW1 = b.T @ gpre
    gb = gpre @ W1.T
    n = np.arange(1, W1.shape[0] + 1, dtype=np.float64).reshape(1, -1)
    k = n * np.pi / cutoff
    rr = np.where(r > 0.0, r, 1.0).reshape(-1, 1)
    db = np.sqrt(2.0 / cutoff) * (k * np.cos(k * rr) / rr - np.sin(k * rr) / rr ** 2)
    dr = np.where(r > 0.0, (gb * db).sum(axis=1), 0.0)
    gvec = v * (dr / np.where(r > 0.0, r, 1.0)).reshape(-1, 1)
    return gvec, gW1, gW2


# ------------------------------------------------ channel mixing ('uvw') ---
#
# NVIDIA's SE(3)-Transformer blog, section "TFN fusion": the pairwise degree
# convolutions of a layer are summed per output degree, and the fused variants
# concatenate degrees so that the channel contractions become dense products
# whose sizes are multiples of 16, for the tensor cores.  The dense part is a
# per-irrep channel mixing.  For an instruction (i, o) between an input and an
# output irrep of the same l and parity, with its own matrix W [mul_in, mul_out]:
#     out[n, o, m, w] += sum_u x[n, i, m, u] W[u, w]          (m = -l..l)
# Readings (the pages give no formula): no normalisation factor (the caller
# scales W); outputs that no instruction reaches are zero; the weights of the
# instructions are stored one after another, each row-major [mul_in][mul_out].
# numpy's einsum (a library contraction) is the only step beyond loops.

def _blocks(irreps):
    off, res = 0, []
    for mul, l, p in irreps:
        res.append((off, mul, l, p))
        off += mul * (2 * l + 1)
    return res


def linear_instructions(irreps_in: str, irreps_out: str):
    """Every (i, o) pair of input and output irreps with the same l and parity,
    input-major."""
    a, b = parse_irreps(irreps_in), parse_irreps(irreps_out)
    return [(i, o) for i, (_, li, pi) in enumerate(a) for o, (_, lo, po) in enumerate(b)
            if li == lo and pi == po]


def _linear_layout(irreps_in, irreps_out, instr):
    a, b = _blocks(parse_irreps(irreps_in)), _blocks(parse_irreps(irreps_out))
    res, offw = [], 0
    for i, o in instr:
        (oi, mi, li, pi), (oo, mo, lo, po) = a[i], b[o]
        if li != lo or pi != po:
            raise ValueError(f"instruction ({i}, {o}) joins different irreps")
        res.append((oi, mi, oo, mo, 2 * li + 1, offw))
        offw += mi * mo
    dim_in = sum(m * (2 * l + 1) for m, l, _ in parse_irreps(irreps_in))
    dim_out = sum(m * (2 * l + 1) for m, l, _ in parse_irreps(irreps_out))
    return res, dim_in, dim_out, offw


def linear_forward(irreps_in: str, irreps_out: str, instr, x, W) -> np.ndarray:
    lay, dim_in, dim_out, nw = _linear_layout(irreps_in, irreps_out, instr)
    x, W = _f64(x), _f64(W)
    if x.shape[1] != dim_in or W.shape != (nw,):
        raise ValueError("x / W do not match the irreps")
    out = np.zeros((x.shape[0], dim_out))
    for oi, mi, oo, mo, d, ow in lay:
        xb = x[:, oi:oi + d * mi].reshape(-1, d, mi)
        Wj = W[ow:ow + mi * mo].reshape(mi, mo)
        out[:, oo:oo + d * mo] += np.einsum("nmu,uw->nmw", xb, Wj).reshape(-1, d * mo)
    return out


def linear_backward(irreps_in: str, irreps_out: str, instr, x, W, g):
    """(dL/dx, dL/dW) for the cotangent g = dL/dout."""
    lay, dim_in, dim_out, nw = _linear_layout(irreps_in, irreps_out, instr)
    x, W, g = _f64(x), _f64(W), _f64(g)
    gx, gW = np.zeros_like(x), np.zeros(nw)
    for oi, mi, oo, mo, d, ow in lay:
        xb = x[:, oi:oi + d * mi].reshape(-1, d, mi)
        gb = g[:, oo:oo + d * mo].reshape(-1, d, mo)
        Wj = W[ow:ow + mi * mo].reshape(mi, mo)
        gx[:, oi:oi + d * mi] += np.einsum("nmw,uw->nmu", gb, Wj).reshape(-1, d * mi)
        gW[ow:ow + mi * mo] += np.einsum("nmu,nmw->uw", xb, gb).ravel()
    return gx, gW


def tp_uvw_forward(irreps_in1: str, irreps_in2: str, irreps_out: str, x, y, W) -> np.ndarray:
    """Tensor product with full channel mixing per path ('uvw', one weight
    matrix per path shared by all rows):
        out[b, k, m3, w] = sum_paths->k sum_u sum_{m1,m2}
                           C[m1, m2, m3] x[b, i1, m1, u] y[b, i2, m2] W_p[u, w]
    Paths: every parity-allowed (i1, i2, k) with mul(in2) = 1, in1-major, then
    in2, then out (the output multiplicity may differ from in1's).  W holds
    the paths' [mul1, mul_out] matrices one after another."""
    a, b, c = (_blocks(parse_irreps(s)) for s in (irreps_in1, irreps_in2, irreps_out))
    x, y, W = _f64(x), _f64(y), _f64(W)
    out = np.zeros((x.shape[0], sum(m * (2 * l + 1) for _, m, l, _ in c)))
    ow = 0
    for o1, m1, l1, p1 in a:
        for o2, m2, l2, p2 in b:
            for o3, m3, l3, p3 in c:
                if not (abs(l1 - l2) <= l3 <= l1 + l2 and p3 == p1 * p2 and m2 == 1):
                    continue
                C = cg_real(l1, l2, l3)
                xb = x[:, o1:o1 + (2 * l1 + 1) * m1].reshape(-1, 2 * l1 + 1, m1)
                yb = y[:, o2:o2 + 2 * l2 + 1]
                Wp = W[ow:ow + m1 * m3].reshape(m1, m3)
                ow += m1 * m3
                out[:, o3:o3 + (2 * l3 + 1) * m3] += np.einsum(
                    "ijk,biu,bj,uw->bkw", C, xb, yb, Wp).reshape(x.shape[0], -1)
    if W.shape != (ow,):
        raise ValueError("W does not match the paths")
    return out


def tp_uvw_backward(irreps_in1: str, irreps_in2: str, irreps_out: str, x, y, W, g):
    """(dL/dx, dL/dy, dL/dW) of ``tp_uvw_forward`` for dL/dout = g: the
    contraction with one operand left out at a time (W summed over rows)."""
    a, b, c = (_blocks(parse_irreps(s)) for s in (irreps_in1, irreps_in2, irreps_out))
    x, y, W, g = _f64(x), _f64(y), _f64(W), _f64(g)
    gx, gy, gW = np.zeros_like(x), np.zeros_like(y), np.zeros_like(W)
    B, ow = x.shape[0], 0
    for o1, m1, l1, p1 in a:
        for o2, m2, l2, p2 in b:
            for o3, m3, l3, p3 in c:
                if not (abs(l1 - l2) <= l3 <= l1 + l2 and p3 == p1 * p2 and m2 == 1):
                    continue
                C = cg_real(l1, l2, l3)
                xb = x[:, o1:o1 + (2 * l1 + 1) * m1].reshape(B, 2 * l1 + 1, m1)
                yb = y[:, o2:o2 + 2 * l2 + 1]
                gb = g[:, o3:o3 + (2 * l3 + 1) * m3].reshape(B, 2 * l3 + 1, m3)
                Wp = W[ow:ow + m1 * m3].reshape(m1, m3)
                gx[:, o1:o1 + (2 * l1 + 1) * m1] += np.einsum(
                    "ijk,bj,uw,bkw->biu", C, yb, Wp, gb).reshape(B, -1)
                gy[:, o2:o2 + 2 * l2 + 1] += np.einsum("ijk,biu,uw,bkw->bj", C, xb, Wp, gb)
                gW[ow:ow + m1 * m3] += np.einsum("ijk,biu,bj,bkw->uw", C, xb, yb, gb).ravel()
                ow += m1 * m3
    return gx, gy, gW
