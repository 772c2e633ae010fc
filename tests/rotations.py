"""Rotation helpers for the equivariance pins (test code only).

A Wigner-D matrix of degree l is not typed in from a formula: it is fitted by
least squares from spherical harmonics of rotated points, Y_l(R r) = D_l Y_l(r),
using the oracle's harmonics (themselves pinned against scipy), and is checked
to be orthogonal.
"""
import numpy as np


def random_rotation(rng) -> np.ndarray:
    q = rng.standard_normal(4)
    q /= np.linalg.norm(q)
    a, b, c, d = q
    return np.array([
        [a * a + b * b - c * c - d * d, 2 * (b * c - a * d), 2 * (b * d + a * c)],
        [2 * (b * c + a * d), a * a - b * b + c * c - d * d, 2 * (c * d - a * b)],
        [2 * (b * d - a * c), 2 * (c * d + a * b), a * a - b * b - c * c + d * d],
    ])


def wigner_d(sh, lmax: int, R: np.ndarray, rng) -> list:
    """[D_0, ..., D_lmax] fitted from sh(lmax, points)."""
    pts = rng.standard_normal((64, 3))
    Y = sh(lmax, pts)
    YR = sh(lmax, pts @ R.T)
    Ds = []
    for l in range(lmax + 1):
        s = slice(l * l, (l + 1) * (l + 1))
        # YR[:, s] = Y[:, s] @ D^T
        Dt, *_ = np.linalg.lstsq(Y[:, s], YR[:, s], rcond=None)
        D = Dt.T
        assert np.abs(D @ D.T - np.eye(2 * l + 1)).max() < 1e-10
        Ds.append(D)
    return Ds


def rotate_features(x: np.ndarray, irreps, Ds, parity_sign: int = 1) -> np.ndarray:
    """Apply D_l to every irrep block of rows x[..., dim] laid out [2l+1][mul];
    with parity_sign = -1 also multiply odd blocks by -1 (inversion)."""
    out = np.empty_like(x)
    off = 0
    for mul, l, p in irreps:
        d = 2 * l + 1
        blk = x[..., off:off + d * mul].reshape(x.shape[:-1] + (d, mul))
        r = np.einsum("ij,...jm->...im", Ds[l], blk)
        if parity_sign == -1 and p == -1:
            r = -r
        out[..., off:off + d * mul] = r.reshape(x.shape[:-1] + (d * mul,))
        off += d * mul
    return out
