"""Pins of the oracle's real spherical harmonics and their derivatives (CPU).

What fixes them: the closed forms for l <= 2, scipy's complex spherical
harmonics taken to the real basis (a library routine), the addition theorem
sum_m Y_lm^2 = 2l+1, orthogonality on the sphere by quadrature, parity, scale
invariance, and central finite differences for the vector-Jacobian and
Jacobian-vector products.
"""
import math

import numpy as np
import pytest

import oracle as O


def _unit(rng, n):
    v = rng.standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


def test_closed_forms_l_le_2():
    rng = np.random.default_rng(0)
    u = _unit(rng, 50)
    x, y, z = u.T
    Y = O.sh(2, u)
    s3, s5, s15 = math.sqrt(3), math.sqrt(5), math.sqrt(15)
    ref = np.stack([np.ones_like(x), s3 * y, s3 * z, s3 * x, s15 * x * y, s15 * y * z,
                    s5 / 2 * (3 * z * z - 1), s15 * x * z, s15 / 2 * (x * x - y * y)], axis=1)
    assert np.abs(Y - ref).max() < 1e-14


def test_matches_scipy_real_basis():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(1)
    u = _unit(rng, 40)
    theta = np.arccos(np.clip(u[:, 2], -1, 1))
    phi = np.arctan2(u[:, 1], u[:, 0])
    lmax = 6
    Y = O.sh(lmax, u)
    for l in range(lmax + 1):
        for m in range(-l, l + 1):
            c = sp.sph_harm_y(l, abs(m), theta, phi)  # orthonormal, Condon-Shortley
            if m == 0:
                ref = c.real
            elif m > 0:
                ref = math.sqrt(2) * (-1) ** m * c.real
            else:
                ref = math.sqrt(2) * (-1) ** m * c.imag
            ref = ref * math.sqrt(4 * math.pi)
            assert np.abs(Y[:, l * l + m + l] - ref).max() < 1e-12, (l, m)


def test_addition_theorem_parity_scale():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((30, 3))
    lmax = 6
    Y = O.sh(lmax, v)
    for l in range(lmax + 1):
        s = slice(l * l, (l + 1) ** 2)
        assert np.abs((Y[:, s] ** 2).sum(1) - (2 * l + 1)).max() < 1e-12
        assert np.abs(O.sh(lmax, -v)[:, s] - (-1) ** l * Y[:, s]).max() < 1e-12
    assert np.abs(O.sh(lmax, 3.7 * v) - Y).max() < 1e-12


def test_orthogonal_on_sphere():
    lmax = 4
    zs, wz = np.polynomial.legendre.leggauss(20)
    nphi = 24
    phi = 2 * math.pi * np.arange(nphi) / nphi
    Z, P = np.meshgrid(zs, phi, indexing="ij")
    W = np.repeat(wz, nphi) * (2 * math.pi / nphi)
    s = np.sqrt(1 - Z.ravel() ** 2)
    pts = np.stack([s * np.cos(P.ravel()), s * np.sin(P.ravel()), Z.ravel()], 1)
    Y = O.sh(lmax, pts)
    G = (Y * W[:, None]).T @ Y / (4 * math.pi)
    assert np.abs(G - np.eye(G.shape[0])).max() < 1e-12


@pytest.mark.parametrize("lmax", [1, 3, 5])
def test_vjp_jvp_finite_differences(lmax):
    rng = np.random.default_rng(3 + lmax)
    v = rng.standard_normal((12, 3))
    gy = rng.standard_normal((12, (lmax + 1) ** 2))
    t = rng.standard_normal((12, 3))
    h = 1e-6
    fd = (O.sh(lmax, v + h * t) - O.sh(lmax, v - h * t)) / (2 * h)
    jvp = O.sh_jvp(lmax, v, t)
    assert np.abs(jvp - fd).max() < 1e-7 * max(1.0, np.abs(fd).max())
    vjp = O.sh_vjp(lmax, v, gy)
    # adjoint identity per edge: <J^T gy, t> = <gy, J t>
    assert np.abs((vjp * t).sum(1) - (gy * jvp).sum(1)).max() < 1e-12
    # gradient is orthogonal to the radial direction (Y depends on r/|r| only)
    assert np.abs((vjp * v).sum(1)).max() < 1e-11


@pytest.mark.parametrize("lmax", [0, 1, 2, 3, 6])
def test_hvp_finite_differences_symmetry_homogeneity(lmax):
    """Second derivatives of s(r) = gy . Y(r): central differences of the
    (separately pinned) vector-Jacobian product, symmetry of the Hessian, and
    Euler's identity for a function of degree 0 in r, H r = -grad s."""
    rng = np.random.default_rng(11 + lmax)
    v = rng.standard_normal((10, 3)) * rng.uniform(0.5, 3.0, (10, 1))
    gy = rng.standard_normal((10, (lmax + 1) ** 2))
    a, b = rng.standard_normal((10, 3)), rng.standard_normal((10, 3))
    h = 1e-5
    fd = (O.sh_vjp(lmax, v + h * a, gy) - O.sh_vjp(lmax, v - h * a, gy)) / (2 * h)
    Ha = O.sh_hvp(lmax, v, gy, a)
    scale = max(1.0, np.abs(fd).max())
    assert np.abs(Ha - fd).max() < 1e-7 * scale
    Hb = O.sh_hvp(lmax, v, gy, b)
    assert np.abs((Ha * b).sum(1) - (Hb * a).sum(1)).max() < 1e-11 * scale
    Hv = O.sh_hvp(lmax, v, gy, v)
    assert np.abs(Hv + O.sh_vjp(lmax, v, gy)).max() < 1e-11 * scale
    # degree -2 in |r|: H(2 r) = H(r) / 4
    assert np.abs(O.sh_hvp(lmax, 2 * v, gy, a) - Ha / 4).max() < 1e-12 * scale


def test_hvp_closed_form_l1():
    """l = 1: gy . Y(r) = sqrt(3) (c . r) / |r| with c = (gy_x, gy_y, gy_z) =
    (gy[3], gy[1], gy[2]); its Hessian is
    [-(c r^T + r c^T) - (c.r) I + 3 (c.r) r r^T / |r|^2] / |r|^3."""
    rng = np.random.default_rng(5)
    v = rng.standard_normal((8, 3))
    gy = rng.standard_normal((8, 4))
    t = rng.standard_normal((8, 3))
    got = O.sh_hvp(1, v, gy, t)
    for e in range(8):
        r, c = v[e], math.sqrt(3) * np.array([gy[e, 3], gy[e, 1], gy[e, 2]])
        rho = np.linalg.norm(r)
        cr = c @ r
        H = (-(np.outer(c, r) + np.outer(r, c)) - cr * np.eye(3)
             + 3 * cr * np.outer(r, r) / rho ** 2) / rho ** 3
        assert np.abs(got[e] - H @ t[e]).max() < 1e-13
