"""Pins of the oracle's Clebsch-Gordan coefficients (CPU only).

What fixes them: sympy's CG table (a library routine independent of the
oracle's Racah sum), textbook closed forms, unitarity, the stated sign
convention, and equivariance under rotations with Wigner-D matrices fitted from
the (separately pinned) spherical harmonics.
"""
import itertools
import math

import numpy as np
import pytest

import oracle as O
from tests.rotations import random_rotation, wigner_d


def _triples(lmax):
    for l1, l2, l3 in itertools.product(range(lmax + 1), repeat=3):
        if abs(l1 - l2) <= l3 <= l1 + l2:
            yield l1, l2, l3


def test_complex_cg_matches_sympy():
    sympy = pytest.importorskip("sympy")
    from sympy.physics.quantum.cg import CG

    worst = 0.0
    for l1, l2, l3 in _triples(3):
        for m1 in range(-l1, l1 + 1):
            for m2 in range(-l2, l2 + 1):
                m3 = m1 + m2
                if abs(m3) > l3:
                    continue
                ref = float(CG(l1, m1, l2, m2, l3, m3).doit().evalf(30))
                worst = max(worst, abs(O.cg_complex(l1, m1, l2, m2, l3, m3) - ref))
    assert worst < 1e-14


def test_complex_cg_textbook_values():
    # Standard table entries for 1 x 1 coupling.
    assert O.cg_complex(1, 1, 1, -1, 2, 0) == pytest.approx(1 / math.sqrt(6), abs=1e-15)
    assert O.cg_complex(1, 0, 1, 0, 2, 0) == pytest.approx(math.sqrt(2 / 3), abs=1e-15)
    assert O.cg_complex(1, 1, 1, -1, 0, 0) == pytest.approx(1 / math.sqrt(3), abs=1e-15)
    assert O.cg_complex(1, 0, 1, 0, 0, 0) == pytest.approx(-1 / math.sqrt(3), abs=1e-15)
    assert O.cg_complex(1, 1, 1, -1, 1, 0) == pytest.approx(1 / math.sqrt(2), abs=1e-15)
    assert O.cg_complex(1, 0, 1, 0, 1, 0) == 0.0
    assert O.cg_complex(2, 2, 1, -1, 3, 1) == pytest.approx(1 / math.sqrt(15), abs=1e-15)
    assert O.cg_complex(1, 1, 1, 1, 2, 1) == 0.0  # m3 != m1 + m2


def test_real_cg_unitary():
    for l1, l2, l3 in _triples(4):
        C = O.cg_real(l1, l2, l3).reshape(-1, 2 * l3 + 1)
        assert np.abs(C.T @ C - np.eye(2 * l3 + 1)).max() < 1e-13, (l1, l2, l3)


def test_real_cg_completeness():
    # sum over l3 of C C^T is the identity on the (l1, l2) product space.
    for l1, l2 in itertools.product(range(4), repeat=2):
        acc = np.zeros(((2 * l1 + 1) * (2 * l2 + 1),) * 2)
        for l3 in range(abs(l1 - l2), l1 + l2 + 1):
            C = O.cg_real(l1, l2, l3).reshape(-1, 2 * l3 + 1)
            acc += C @ C.T
        assert np.abs(acc - np.eye(acc.shape[0])).max() < 1e-13


def test_real_cg_closed_forms():
    for l in range(5):
        d = 2 * l + 1
        assert np.allclose(O.cg_real(0, l, l)[0], np.eye(d), atol=1e-15)
        assert np.allclose(O.cg_real(l, 0, l)[:, 0, :], np.eye(d), atol=1e-15)
        assert np.allclose(O.cg_real(l, l, 0)[:, :, 0], np.eye(d) / math.sqrt(d), atol=1e-15)
    # 1 x 1 -> 1 is the Levi-Civita tensor / sqrt 2 in (y, z, x) order.
    eps = np.zeros((3, 3, 3))
    for (i, j, k), s in {(0, 1, 2): 1, (1, 2, 0): 1, (2, 0, 1): 1,
                         (0, 2, 1): -1, (2, 1, 0): -1, (1, 0, 2): -1}.items():
        eps[i, j, k] = s
    assert np.allclose(O.cg_real(1, 1, 1), eps / math.sqrt(2), atol=1e-15)
    # 1 x 1 -> 2: each output component is a symmetric traceless 3x3 matrix.
    C = O.cg_real(1, 1, 2)
    for m in range(5):
        M = C[:, :, m]
        assert np.allclose(M, M.T, atol=1e-15) and abs(np.trace(M)) < 1e-15


def test_real_cg_sign_convention_and_zero_triangle():
    for l1, l2, l3 in _triples(4):
        C = O.cg_real(l1, l2, l3).ravel()
        first = C[np.nonzero(np.abs(C) > 0)[0][0]]
        assert first > 0
    assert not O.cg_real(1, 1, 3).any()
    with pytest.raises(ValueError):
        O.cg_real(7, 0, 7)


def test_real_cg_equivariant():
    rng = np.random.default_rng(11)
    for _ in range(5):
        R = random_rotation(rng)
        Ds = wigner_d(O.sh, 4, R, rng)
        for l1, l2, l3 in _triples(4):
            C = O.cg_real(l1, l2, l3)
            lhs = np.einsum("abc,ai,bj->ijc", C, Ds[l1], Ds[l2])
            rhs = np.einsum("ijk,ck->ijc", C, Ds[l3])
            assert np.abs(lhs - rhs).max() < 1e-10, (l1, l2, l3)


def test_sh_product_projection():
    """sum C[m1,m2,m3] Y_l1 Y_l2 = s sqrt(d1 d2 / d3) <l1 0 l2 0|l3 0> Y_l3 with
    s = +-1 (the path's sign convention); zero when l1+l2+l3 is odd."""
    sympy = pytest.importorskip("sympy")
    from sympy.physics.quantum.cg import CG

    rng = np.random.default_rng(3)
    Y = O.sh(4, rng.standard_normal((20, 3)))
    blk = lambda l: Y[:, l * l:(l + 1) * (l + 1)]
    for l1, l2, l3 in _triples(3):
        lhs = np.einsum("abc,na,nb->nc", O.cg_real(l1, l2, l3), blk(l1), blk(l2))
        c0 = float(CG(l1, 0, l2, 0, l3, 0).doit().evalf(30))
        k = math.sqrt((2 * l1 + 1) * (2 * l2 + 1) / (2 * l3 + 1)) * c0
        if (l1 + l2 + l3) % 2:
            assert np.abs(lhs).max() < 1e-12
        else:
            ok = min(np.abs(lhs - k * blk(l3)).max(), np.abs(lhs + k * blk(l3)).max())
            assert ok < 1e-12, (l1, l2, l3)
