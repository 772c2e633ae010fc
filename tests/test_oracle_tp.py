"""Pins of the oracle's tensor product, convolution, gradients and forces (CPU).

What fixes them: hand-checkable tiny cases (x.y/sqrt3, scalar scaling),
equivariance under random rotations and inversion (< 1e-10 in fp64), the
trilinear adjoint identity, central finite differences of the gradients and of
the double backward, the fused convolution equal to gathered standalone
products summed per receiver, and translation invariance of the forces.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests.rotations import random_rotation, rotate_features, wigner_d

SMALL = ("3x0e+3x1o+3x2e", "0e+1o+2e+3o", "3x0e+3x1o+3x1e+3x2o+3x2e+3x3o+3x3e")
ODD = ("2x0e+2x1o+2x2e+2x3o", "0e+1o+2e+3o", "2x0e+2x1o+2x2e+2x3o")


def _rand(rng, prob, B):
    return (rng.standard_normal((B, prob.dim1)), rng.standard_normal((B, prob.dim2)),
            rng.standard_normal((B, prob.wdim)))


def test_path_enumeration():
    p = O.make_problem(*W.IRREPS_TP16)
    got = [(l1, l2, l3) for (_, _, _, l1, l2, l3, *_r) in p.paths]
    assert got == [(0, 0, 0), (0, 1, 1), (0, 2, 2), (1, 0, 1), (1, 1, 0), (1, 1, 2), (1, 2, 1)]
    assert (p.dim1, p.dim2, p.dimo, p.wdim) == (64, 9, 144, 112)
    p1 = O.make_problem(*W.IRREPS_MACE128)
    assert len(p1.paths) == 24 and (p1.dim1, p1.dimo, p1.wdim) == (1152, 3968, 3072)
    assert len(O.make_problem(*W.IRREPS_TFN32).paths) == 23
    with pytest.raises(ValueError):
        O.parse_irreps("3x1q")


def test_tiny_closed_forms():
    rng = np.random.default_rng(0)
    # 1o x 1o -> 0e, mul 1: out = w (x . y) / sqrt 3 in any consistent basis.
    p = O.make_problem("1x1o", "1o", "1x0e")
    x, y, w = rng.standard_normal((5, 3)), rng.standard_normal((5, 3)), rng.standard_normal((5, 1))
    out = O.tp_forward(p, x, y, w)
    assert np.abs(out[:, 0] - w[:, 0] * (x * y).sum(1) / math.sqrt(3)).max() < 1e-14
    # 1o x 1o -> 1e: out = w (x cross y) / sqrt 2 in (y, z, x) component order.
    p = O.make_problem("1x1o", "1o", "1x1e")
    out = O.tp_forward(p, x, y, w)
    perm = [2, 0, 1]  # (y,z,x) -> (x,y,z)
    cr = np.cross(x[:, perm], y[:, perm])[:, [1, 2, 0]]
    assert np.abs(out - w * cr / math.sqrt(2)).max() < 1e-14
    # scalar in2: 4x2e (x) 0e -> 4x2e multiplies by y0 w_u.
    p = O.make_problem("4x2e", "0e", "4x2e")
    x, y, w = rng.standard_normal((3, 20)), rng.standard_normal((3, 1)), rng.standard_normal((3, 4))
    out = O.tp_forward(p, x, y, w)
    ref = x.reshape(3, 5, 4) * y[:, :, None] * w[:, None, :]
    assert np.abs(out - ref.reshape(3, 20)).max() < 1e-14


@pytest.mark.parametrize("irreps", [SMALL, ODD])
def test_equivariance_rotation_and_inversion(irreps):
    rng = np.random.default_rng(1)
    prob = O.make_problem(*irreps)
    x, _, w = _rand(rng, prob, 6)
    v = rng.standard_normal((6, 3))
    y = O.sh(3, v)
    out = O.tp_forward(prob, x, y, w)
    for _ in range(20):
        R = random_rotation(rng)
        Ds = wigner_d(O.sh, 3, R, rng)
        xr = rotate_features(x, prob.in1, Ds)
        yr = O.sh(3, v @ R.T)
        got = O.tp_forward(prob, xr, yr, w)
        assert np.abs(got - rotate_features(out, prob.out, Ds)).max() < 1e-10
    eye = [np.eye(2 * l + 1) for l in range(4)]
    got = O.tp_forward(prob, rotate_features(x, prob.in1, eye, -1), O.sh(3, -v), w)
    assert np.abs(got - rotate_features(out, prob.out, eye, -1)).max() < 1e-12


def test_adjoint_identity_and_finite_differences():
    rng = np.random.default_rng(2)
    prob = O.make_problem(*SMALL)
    x, y, w = _rand(rng, prob, 4)
    g = rng.standard_normal((4, prob.dimo))
    gx, gy, gw = O.tp_backward(prob, x, y, w, g)
    s = (g * O.tp_forward(prob, x, y, w)).sum()
    assert abs((gx * x).sum() - s) < 1e-10 * abs(s)
    assert abs((gy * y).sum() - s) < 1e-10 * abs(s)
    assert abs((gw * w).sum() - s) < 1e-10 * abs(s)
    h = 1e-6
    for arg, grad in ((0, gx), (1, gy), (2, gw)):
        t = rng.standard_normal(grad.shape)
        a = [x, y, w]
        ap, am = list(a), list(a)
        ap[arg] = a[arg] + h * t
        am[arg] = a[arg] - h * t
        fd = ((g * O.tp_forward(prob, *ap)).sum() - (g * O.tp_forward(prob, *am)).sum()) / (2 * h)
        assert abs(fd - (grad * t).sum()) < 1e-7 * max(1.0, abs(fd))


def test_shared_weights_backward_sums_rows():
    rng = np.random.default_rng(3)
    prob = O.make_problem(*ODD)
    x, y, _ = _rand(rng, prob, 5)
    w1 = rng.standard_normal(prob.wdim)
    g = rng.standard_normal((5, prob.dimo))
    out = O.tp_forward(prob, x, y, w1)
    assert np.abs(out - O.tp_forward(prob, x, y, np.tile(w1, (5, 1)))).max() < 1e-13
    gw = O.tp_backward(prob, x, y, w1, g)[2]
    gw_rows = O.tp_backward(prob, x, y, np.tile(w1, (5, 1)), g)[2]
    assert np.abs(gw - gw_rows.sum(0)).max() < 1e-12


@pytest.mark.parametrize("shared", [False, True])
def test_double_backward_finite_differences(shared):
    rng = np.random.default_rng(4)
    prob = O.make_problem(*SMALL)
    x, y, w = _rand(rng, prob, 3)
    if shared:  # one weight row for every sample: d_w sums the rows
        w = w[0].copy()
    g = rng.standard_normal((3, prob.dimo))
    ggx, ggy, ggw = (rng.standard_normal(a.shape) for a in (x, y, w))

    def S(x_, y_, w_, g_):
        a, b, c = O.tp_backward(prob, x_, y_, w_, g_)
        return (ggx * a).sum() + (ggy * b).sum() + (ggw * c).sum()

    d = O.tp_double_backward(prob, x, y, w, g, ggx, ggy, ggw)
    h = 1e-6
    args = [x, y, w, g]
    for k in range(4):
        t = rng.standard_normal(args[k].shape)
        ap, am = list(args), list(args)
        ap[k] = args[k] + h * t
        am[k] = args[k] - h * t
        fd = (S(*ap) - S(*am)) / (2 * h)
        assert abs(fd - (d[k] * t).sum()) < 1e-7 * max(1.0, abs(fd)), k


def _small_graph(rng, N=9):
    recv, send = [], []
    for n in range(N):
        if n == 4:
            continue  # an isolated receiver
        for s in rng.choice(N, size=rng.integers(1, 5), replace=False):
            recv.append(n)
            send.append(s)
    return W.make_graph(N, np.array(recv), np.array(send), rng.standard_normal((len(recv), 3)))


def test_conv_equals_gathered_standalone_sum():
    rng = np.random.default_rng(5)
    prob = O.make_problem(*ODD)
    g = _small_graph(rng)
    x = rng.standard_normal((g.N, prob.dim1))
    y = O.sh(3, g.vec)
    w = rng.standard_normal((g.E, prob.wdim))
    out = O.conv_forward(prob, g.rowptr, g.sender, x, y, w, 0.7)
    per_edge = O.tp_forward(prob, x[g.sender], y, w)
    ref = np.zeros((g.N, prob.dimo))
    np.add.at(ref, g.receiver, per_edge)
    assert np.abs(out - 0.7 * ref).max() < 1e-12
    assert not out[4].any()
    sel = O.conv_forward(prob, g.rowptr, g.sender, x, y, w, 0.7, receivers=[2, 6])
    assert np.array_equal(sel[[2, 6]], out[[2, 6]]) and not sel[[0, 1, 3]].any()

    # gradient: scattered standalone gradients
    gout = rng.standard_normal((g.N, prob.dimo))
    gx, gy, gw = O.conv_backward(prob, g.rowptr, g.sender, x, y, w, 0.7, gout)
    ex, ey, ew = O.tp_backward(prob, x[g.sender], y, w, 0.7 * gout[g.receiver])
    rx = np.zeros_like(x)
    np.add.at(rx, g.sender, ex)
    assert np.abs(gx - rx).max() < 1e-12
    assert np.abs(gy - ey).max() < 1e-12 and np.abs(gw - ew).max() < 1e-12
    sx, sy, sw = O.conv_backward(prob, g.rowptr, g.sender, x, y, w, 0.7, gout, nodes=[1, 3],
                                 edges=[0, 5])
    assert np.array_equal(sx[[1, 3]], gx[[1, 3]]) and np.array_equal(sw[[0, 5]], gw[[0, 5]])


def test_conv_double_backward_finite_differences():
    rng = np.random.default_rng(6)
    prob = O.make_problem(*ODD)
    gr = _small_graph(rng, 7)
    x = rng.standard_normal((gr.N, prob.dim1))
    y = rng.standard_normal((gr.E, prob.dim2))
    w = rng.standard_normal((gr.E, prob.wdim))
    g = rng.standard_normal((gr.N, prob.dimo))
    ggx, ggy, ggw = (rng.standard_normal(a.shape) for a in (x, y, w))
    cb = lambda a, b, c, d: O.conv_backward(prob, gr.rowptr, gr.sender, a, b, c, 0.5, d)

    def S(*a):
        r = cb(*a)
        return (ggx * r[0]).sum() + (ggy * r[1]).sum() + (ggw * r[2]).sum()

    d = O.conv_double_backward(prob, gr.rowptr, gr.sender, x, y, w, 0.5, g, ggx, ggy, ggw)
    args, h = [x, y, w, g], 1e-6
    for k in range(4):
        t = rng.standard_normal(args[k].shape)
        ap, am = list(args), list(args)
        ap[k] = args[k] + h * t
        am[k] = args[k] - h * t
        fd = (S(*ap) - S(*am)) / (2 * h)
        assert abs(fd - (d[k] * t).sum()) < 1e-7 * max(1.0, abs(fd)), k


def test_forces_chain_finite_differences():
    """E(pos) = sum c * conv(x, Y(pos[recv] - pos[send]), w): the force chain
    (conv gradient -> SH vjp -> edge_forces) equals -dE/dpos; forces sum to 0."""
    rng = np.random.default_rng(7)
    prob = O.make_problem("2x0e+2x1o", "0e+1o+2e+3o", "2x0e+2x1o")
    pos, gr = W.molecules(rng, 3, 4, 6)
    x = rng.standard_normal((gr.N, prob.dim1))
    w = rng.standard_normal((gr.E, prob.wdim))
    c = rng.standard_normal((gr.N, prob.dimo))

    def energy(p):
        vec = p[gr.receiver] - p[gr.sender]
        return (c * O.conv_forward(prob, gr.rowptr, gr.sender, x, O.sh(3, vec), w, 1.0)).sum()

    vec = pos[gr.receiver] - pos[gr.sender]
    gy = O.conv_backward(prob, gr.rowptr, gr.sender, x, O.sh(3, vec), w, 1.0, c)[1]
    F = O.edge_forces(gr.rowptr, gr.sender, O.sh_vjp(3, vec, gy))
    assert np.abs(F.sum(0)).max() < 1e-10
    h = 1e-6
    for _ in range(3):
        t = rng.standard_normal(pos.shape)
        fd = (energy(pos + h * t) - energy(pos - h * t)) / (2 * h)
        assert abs(fd + (F * t).sum()) < 1e-6 * max(1.0, abs(fd))


def test_force_loss_position_gradient_finite_differences():
    """L(pos) = sum gF * F(pos) for the forces of the chain above.  Its gradient
    in the positions goes through the second derivatives of the SH only (the
    gradient of the energy in Y does not depend on Y): with q_e = gF[send] -
    gF[recv], dL/dr_e = H_e q_e where H_e is the Hessian in r_e of
    gY_e . Y(r_e), and dL/dpos = -edge_forces(dL/dr)."""
    rng = np.random.default_rng(8)
    prob = O.make_problem("2x0e+2x1o+1x2e", "0e+1o+2e+3o", "2x0e+2x1o+1x2e")
    pos, gr = W.molecules(rng, 3, 4, 6)
    x = rng.standard_normal((gr.N, prob.dim1))
    w = rng.standard_normal((gr.E, prob.wdim))
    c = rng.standard_normal((gr.N, prob.dimo))
    gF = rng.standard_normal((gr.N, 3))

    def forces(p):
        vec = p[gr.receiver] - p[gr.sender]
        gy = O.conv_backward(prob, gr.rowptr, gr.sender, x, O.sh(3, vec), w, 1.0, c)[1]
        return O.edge_forces(gr.rowptr, gr.sender, O.sh_vjp(3, vec, gy)), gy

    F, gy = forces(pos)
    vec = pos[gr.receiver] - pos[gr.sender]
    q = gF[gr.sender] - gF[gr.receiver]
    dLdpos = -O.edge_forces(gr.rowptr, gr.sender, O.sh_hvp(3, vec, gy, q))
    assert np.abs(dLdpos.sum(0)).max() < 1e-10  # translation invariance
    h = 1e-5
    for _ in range(3):
        t = rng.standard_normal(pos.shape)
        fd = ((gF * forces(pos + h * t)[0]).sum() - (gF * forces(pos - h * t)[0]).sum()) / (2 * h)
        assert abs(fd - (dLdpos * t).sum()) < 1e-6 * max(1.0, abs(fd))


def test_empty_inputs():
    prob = O.make_problem(*ODD)
    out = O.tp_forward(prob, np.zeros((0, prob.dim1)), np.zeros((0, 16)), np.zeros((0, prob.wdim)))
    assert out.shape == (0, prob.dimo)
    rowptr = np.zeros(4, dtype=np.int32)
    out = O.conv_forward(prob, rowptr, np.zeros(0, np.int32), np.ones((3, prob.dim1)),
                         np.zeros((0, 16)), np.zeros((0, prob.wdim)), 1.0)
    assert out.shape == (3, prob.dimo) and not out.any()
