"""Pins of the oracle's radial network (Bessel basis -> Linear -> SiLU ->
Linear) against facts that do not come from the oracle itself: the
orthonormality of the sine basis on [0, rc] with weight r^2, its values at
r = 0, rc / 2 and rc, the odd part of SiLU, invariance under rotations of the
edge vector, linearity in the last layer and finite differences of the
gradient."""
import numpy as np
import pytest

import oracle as O
from tests.rotations import random_rotation

RC = 5.0


def test_basis_orthonormal_with_weight_r2():
    # integral over [0, rc] of b_n b_m r^2 dr = delta_nm (Gauss-Legendre, exact
    # to rounding for these trigonometric polynomials at 200 nodes)
    t, wq = np.polynomial.legendre.leggauss(200)
    r = 0.5 * RC * (t + 1.0)
    b = O.radial_basis(r, 8, RC)
    G = (b * (0.5 * RC * wq * r * r)[:, None]).T @ b
    assert np.abs(G - np.eye(8)).max() < 1e-12


def test_basis_special_values():
    n = np.arange(1, 9)
    b0 = O.radial_basis(np.array([0.0]), 8, RC)[0]
    assert np.allclose(b0, np.sqrt(2 / RC) * n * np.pi / RC, rtol=0, atol=1e-15)
    # continuity at 0 (sin(x)/x -> 1)
    assert np.abs(O.radial_basis(np.array([1e-7]), 8, RC)[0] - b0).max() < 1e-9
    half = O.radial_basis(np.array([RC / 2]), 8, RC)[0]
    pattern = np.array([1, 0, -1, 0, 1, 0, -1, 0], dtype=float)
    assert np.abs(half - np.sqrt(2 / RC) * pattern / (RC / 2)).max() < 1e-15
    assert np.abs(O.radial_basis(np.array([RC]), 8, RC)[0]).max() < 1e-15


def test_silu_odd_part_and_origin():
    a = np.linspace(-30, 30, 601)
    assert np.abs(O.silu(a) - O.silu(-a) - a).max() < 1e-13
    assert O.silu(np.array([0.0]))[0] == 0.0
    eps = 1e-6
    assert abs((O.silu(np.array([eps]))[0] - O.silu(np.array([-eps]))[0]) / (2 * eps) - 0.5) < 1e-10
    assert abs(O.silu(np.array([40.0]))[0] - 40.0) < 1e-12


def test_forward_worked_case_identity_layers():
    # W1 = W2 = I: w = silu(basis); at r = rc / 2 the basis is sqrt(2/rc) (2/rc) {1,0,-1,0,...}
    vec = np.array([[0.0, 0.0, RC / 2]])
    w, h = O.radial_forward(vec, np.eye(8), np.eye(8), RC)
    c = np.sqrt(2 / RC) * 2 / RC
    s = 1 / (1 + np.exp(-c))
    expect = np.array([c * s, 0, -c * (1 - s), 0, c * s, 0, -c * (1 - s), 0])
    assert np.abs(w[0] - expect).max() < 1e-15
    assert np.abs(h - w).max() == 0.0


def test_forward_invariances():
    rng = np.random.default_rng(11)
    vec = rng.standard_normal((50, 3)) * 2
    W1 = rng.standard_normal((8, 16))
    W2 = rng.standard_normal((16, 24))
    w, _ = O.radial_forward(vec, W1, W2, RC)
    R = random_rotation(rng)
    wr, _ = O.radial_forward(vec @ R.T, W1, W2, RC)
    assert np.abs(wr - w).max() < 1e-12 * np.abs(w).max()
    W2b = rng.standard_normal((16, 24))
    w2, _ = O.radial_forward(vec, W1, W2b, RC)
    w12, _ = O.radial_forward(vec, W1, 2.0 * W2 - W2b, RC)
    assert np.abs(w12 - (2.0 * w - w2)).max() < 1e-12 * np.abs(w12).max()
    # chunking does not change the result beyond the matmul's rounding order
    wc, _ = O.radial_forward(vec, W1, W2, RC, chunk=7)
    assert np.abs(wc - w).max() < 1e-14 * np.abs(w).max()


def test_forward_shape_errors():
    with pytest.raises(ValueError):
        O.radial_forward(np.ones((2, 3)), np.ones((8, 4)), np.ones((5, 6)))


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(12)
    E, nb, hid, no = 4, 5, 6, 7
    vec = rng.standard_normal((E, 3)) * 1.5
    W1 = rng.standard_normal((nb, hid))
    W2 = rng.standard_normal((hid, no))
    g = rng.standard_normal((E, no))
    gv, g1, g2 = O.radial_backward(vec, W1, W2, g, RC)

    def L(v, a, b):
        return float((O.radial_forward(v, a, b, RC)[0] * g).sum())

    eps = 1e-6
    for arr, grad, name in ((vec, gv, "vec"), (W1, g1, "W1"), (W2, g2, "W2")):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [p if arr is t else t for t in (vec, W1, W2)]
            args_m = [m if arr is t else t for t in (vec, W1, W2)]
            fd[idx] = (L(*args_p) - L(*args_m)) / (2 * eps)
        assert np.abs(fd - grad).max() < 1e-6 * max(1.0, np.abs(grad).max()), name


def test_backward_zero_length_edge():
    gv, _, _ = O.radial_backward(np.zeros((1, 3)), np.ones((8, 4)), np.ones((4, 3)),
                                 np.ones((1, 3)), RC)
    assert np.array_equal(gv, np.zeros((1, 3)))
