"""Pins of the oracle's per-irrep channel mixing and of the 'uvw' tensor
product (CPU).

What fixes them: hand-computed small cases written as explicit loops, the
identity matrix, equivariance under fitted Wigner-D rotations and inversion,
exact adjoint identities of a bilinear map, and the reduction of 'uvw' with
diagonal path matrices to the 'uvu' product of the C oracle (pinned on its
own in test_oracle_tp.py).
"""
import numpy as np
import pytest

import oracle as O
from tests.rotations import random_rotation, rotate_features, wigner_d

LIN = ("16x0e+8x1o+4x2e+8x1o", "8x0e+16x1o+4x2e")


def _w(rng, ins, outs, instr):
    a, b = O.parse_irreps(ins), O.parse_irreps(outs)
    return rng.standard_normal(sum(a[i][0] * b[o][0] for i, o in instr))


def test_instructions_pair_equal_irreps():
    assert O.linear_instructions(*LIN) == [(0, 0), (1, 1), (2, 2), (3, 1)]
    assert O.linear_instructions("4x0e+4x1o", "4x0o+4x1e") == []


def test_hand_loops():
    """2x1o -> 3x1o with W [2, 3]: out[m, w] = sum_u x[m, u] W[u, w], written
    as plain loops over the row layout [2l+1][mul]."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 6))
    W = rng.standard_normal(6)
    out = O.linear_forward("2x1o", "3x1o", [(0, 0)], x, W)
    ref = np.zeros((2, 9))
    for n in range(2):
        for m in range(3):
            for w in range(3):
                for u in range(2):
                    ref[n, m * 3 + w] += x[n, m * 2 + u] * W[u * 3 + w]
    assert np.abs(out - ref).max() < 1e-15
    # two instructions into one output add; an unreached output stays zero
    x2 = rng.standard_normal((2, 2 + 1))
    W2 = rng.standard_normal(2 * 1 + 1 * 1)
    out2 = O.linear_forward("2x0e+1x0e", "1x0e+1x1o", [(0, 0), (1, 0)], x2, W2)
    assert np.abs(out2[:, 0] - (x2[:, 0] * W2[0] + x2[:, 1] * W2[1] + x2[:, 2] * W2[2])).max() < 1e-15
    assert not out2[:, 1:].any()


def test_identity_matrices():
    rng = np.random.default_rng(1)
    ir = "5x0e+3x1o+2x2e"
    x = rng.standard_normal((4, O.irreps_dim(O.parse_irreps(ir))))
    instr = O.linear_instructions(ir, ir)
    W = np.concatenate([np.eye(m).ravel() for m, _, _ in O.parse_irreps(ir)])
    assert np.abs(O.linear_forward(ir, ir, instr, x, W) - x).max() == 0


def test_equivariance_rotation_and_inversion():
    rng = np.random.default_rng(2)
    instr = O.linear_instructions(*LIN)
    a, b = O.parse_irreps(LIN[0]), O.parse_irreps(LIN[1])
    x = rng.standard_normal((5, O.irreps_dim(a)))
    W = _w(rng, *LIN, instr)
    out = O.linear_forward(*LIN, instr, x, W)
    for _ in range(5):
        Ds = wigner_d(O.sh, 2, random_rotation(rng), rng)
        got = O.linear_forward(*LIN, instr, rotate_features(x, a, Ds), W)
        assert np.abs(got - rotate_features(out, b, Ds)).max() < 1e-12
    eye = [np.eye(2 * l + 1) for l in range(3)]
    got = O.linear_forward(*LIN, instr, rotate_features(x, a, eye, -1), W)
    assert np.abs(got - rotate_features(out, b, eye, -1)).max() < 1e-14


def test_backward_adjoints_and_finite_differences():
    rng = np.random.default_rng(3)
    instr = O.linear_instructions(*LIN)
    a, b = O.parse_irreps(LIN[0]), O.parse_irreps(LIN[1])
    x = rng.standard_normal((6, O.irreps_dim(a)))
    W = _w(rng, *LIN, instr)
    g = rng.standard_normal((6, O.irreps_dim(b)))
    gx, gW = O.linear_backward(*LIN, instr, x, W, g)
    s = (g * O.linear_forward(*LIN, instr, x, W)).sum()
    # bilinear in (x, W): <g, f(x, W)> = <f_x^T g, x> = <f_W^T g, W>
    assert abs((gx * x).sum() - s) < 1e-11 * abs(s)
    assert abs((gW * W).sum() - s) < 1e-11 * abs(s)
    h = 1e-6
    t = rng.standard_normal(W.shape)
    fd = ((g * O.linear_forward(*LIN, instr, x, W + h * t)).sum()
          - (g * O.linear_forward(*LIN, instr, x, W - h * t)).sum()) / (2 * h)
    assert abs(fd - (gW * t).sum()) < 1e-8 * max(1.0, abs(fd))


UVW = ("4x0e+4x1o+4x2e", "0e+1o+2e+3o", "4x0e+4x1o+4x1e+4x2o+4x2e+4x3o+4x3e")


def test_uvw_with_diagonal_matrices_is_uvu():
    """W_p = diag(w_p) reduces 'uvw' to the 'uvu' product with the shared
    weight row (w_p) -- computed by the C oracle's own loops."""
    rng = np.random.default_rng(4)
    prob = O.make_problem(*UVW)
    x = rng.standard_normal((7, prob.dim1))
    y = O.sh(3, rng.standard_normal((7, 3)))
    w = rng.standard_normal(prob.wdim)
    W = np.concatenate([np.diag(w[p[10]:p[10] + p[6]]).ravel() for p in prob.paths])
    ref = O.tp_forward(prob, x, y, w)  # shared row: broadcast by the oracle
    got = O.tp_uvw_forward(*UVW, x, y, W)
    assert np.abs(got - ref).max() < 1e-13 * np.abs(ref).max()


def test_uvw_output_channels_and_equivariance():
    """mul_out != mul_in: with W_p = a_p (1 x 2) on one channel, output channel
    k is a_p[k] times the one-channel 'uvu' product; rotations commute."""
    rng = np.random.default_rng(5)
    ins = ("1x1o+1x2e", "0e+1o+2e", "2x1o+2x2e")
    prob = O.make_problem("1x1o+1x2e", "0e+1o+2e", "1x1o+1x2e")
    x = rng.standard_normal((3, prob.dim1))
    y = O.sh(2, rng.standard_normal((3, 3)))
    A = rng.standard_normal((len(prob.paths), 2))
    got = O.tp_uvw_forward(*ins, x, y, A.ravel())
    for k in range(2):
        ref = O.tp_forward(prob, x, y, A[:, k].copy())
        blocks = [got[:, 0:6].reshape(3, 3, 2)[:, :, k], got[:, 6:16].reshape(3, 5, 2)[:, :, k]]
        assert np.abs(np.concatenate(blocks, 1) - ref).max() < 1e-13
    v = rng.standard_normal((3, 3))
    out = O.tp_uvw_forward(*ins, x, O.sh(2, v), A.ravel())
    R = random_rotation(rng)
    Ds = wigner_d(O.sh, 2, R, rng)
    got = O.tp_uvw_forward(*ins, rotate_features(x, O.parse_irreps(ins[0]), Ds),
                           O.sh(2, v @ R.T), A.ravel())
    assert np.abs(got - rotate_features(out, O.parse_irreps(ins[2]), Ds)).max() < 1e-12


def test_shape_errors():
    with pytest.raises(ValueError):
        O.linear_forward("2x0e", "2x1o", [(0, 0)], np.zeros((1, 2)), np.zeros(4))
    with pytest.raises(ValueError):
        O.linear_forward("2x0e", "2x0e", [(0, 0)], np.zeros((1, 2)), np.zeros(3))


def test_uvw_backward_adjoints_and_finite_differences():
    """The 'uvw' product is linear in x, in y and in W: <g, f> equals each of
    <f_x^T g, x>, <f_y^T g, y>, <f_W^T g, W>; central differences in all three."""
    rng = np.random.default_rng(6)
    ins = ("3x0e+3x1o+3x2e", "0e+1o+2e", "2x0e+4x1o+2x1e+3x2e")
    a = O.parse_irreps(ins[0])
    # the same path list at 3 output channels; one [3, mul_out] matrix per path
    prob = O.make_problem("3x0e+3x1o+3x2e", "0e+1o+2e", "3x0e+3x1o+3x1e+3x2e")
    outs = {(l, p): m for m, l, p in O.parse_irreps(ins[2])}
    nW = sum(3 * outs[(path[5], prob.out[path[2]][2])] for path in prob.paths)
    x = rng.standard_normal((4, O.irreps_dim(a)))
    y = O.sh(2, rng.standard_normal((4, 3)))
    W = rng.standard_normal(nW)
    g = rng.standard_normal((4, O.irreps_dim(O.parse_irreps(ins[2]))))
    f = lambda x_, y_, W_: O.tp_uvw_forward(*ins, x_, y_, W_)
    gx, gy, gW = O.tp_uvw_backward(*ins, x, y, W, g)
    s = (g * f(x, y, W)).sum()
    for d, v in ((gx, x), (gy, y), (gW, W)):
        assert abs((d * v).sum() - s) < 1e-11 * abs(s)
    h = 1e-6
    for k, (d, v) in enumerate(((gx, x), (gy, y), (gW, W))):
        t = rng.standard_normal(v.shape)
        args_p, args_m = [x, y, W], [x, y, W]
        args_p[k] = v + h * t
        args_m[k] = v - h * t
        fd = ((g * f(*args_p)).sum() - (g * f(*args_m)).sum()) / (2 * h)
        assert abs(fd - (d * t).sum()) < 1e-8 * max(1.0, abs(fd))
