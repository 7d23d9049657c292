"""Pins for the oracle's real spherical harmonics (CPU only)."""
import json
import os
from math import pi, sqrt

import numpy as np
import pytest

from oracle import sh

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_dirs(n, seed):
    v = np.random.default_rng(seed).standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


def test_page_printed_constants():
    """Y00 and the l = 1 triple printed on the Batmobile blog."""
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    n = _random_dirs(50, 0)
    Y = sh.real_sh(n * 3.7)  # scale must not matter
    assert np.allclose(Y[:, 0], g["Y00"], rtol=0, atol=1e-15)
    c = g["l1_coefficient"]
    comp = {"x": n[:, 0], "y": n[:, 1], "z": n[:, 2]}
    where = {"Y10": sh.sh_index(1, 0), "Y11c": sh.sh_index(1, 1), "Y11s": sh.sh_index(1, -1)}
    for name, (axis, sign) in g["l1_components"].items():
        assert np.allclose(Y[:, where[name]], sign * c * comp[axis], rtol=0, atol=1e-15)


def test_matches_scipy_complex_harmonics():
    """Real Y from scipy's complex Y (CS phase): sqrt2 Re / sqrt2 Im."""
    from scipy.special import sph_harm_y

    n = _random_dirs(200, 1)
    theta = np.arccos(np.clip(n[:, 2], -1, 1))
    phi = np.arctan2(n[:, 1], n[:, 0])
    Y = sh.real_sh(n)
    for l in range(4):
        for m in range(-l, l + 1):
            yc = sph_harm_y(l, abs(m), theta, phi)
            if m == 0:
                ref = yc.real
            elif m > 0:
                ref = sqrt(2.0) * yc.real
            else:
                ref = sqrt(2.0) * yc.imag
            assert np.allclose(Y[:, sh.sh_index(l, m)], ref, rtol=0, atol=1e-13), (l, m)


def test_orthonormal_by_quadrature():
    """Gauss-Legendre (cos theta) x uniform phi: exact for degree <= 6."""
    t, wt = np.polynomial.legendre.leggauss(8)
    nphi = 16
    phi = 2 * pi * np.arange(nphi) / nphi
    T, P = np.meshgrid(t, phi, indexing="ij")
    s = np.sqrt(1 - T ** 2)
    n = np.stack([s * np.cos(P), s * np.sin(P), T], axis=-1).reshape(-1, 3)
    w = (wt[:, None] * np.full(nphi, 2 * pi / nphi)[None, :]).reshape(-1)
    Y = sh.real_sh(n)
    gram = Y.T @ (Y * w[:, None])
    assert np.allclose(gram, np.eye(16), atol=1e-13)


def test_z_axis_only_m0_survives():
    """E2Former-V2 Lemma 4.1: along z only m = 0 is nonzero."""
    Y = sh.real_sh(np.array([[0.0, 0.0, 2.5]]))[0]
    for l in range(4):
        for m in range(-l, l + 1):
            want = sqrt((2 * l + 1) / (4 * pi)) if m == 0 else 0.0
            assert abs(Y[sh.sh_index(l, m)] - want) < 1e-14


def test_addition_theorem():
    """sum_m Y_lm(a) Y_lm(b) = (2l+1)/(4pi) P_l(a.b), P_l written out."""
    a, b = _random_dirs(100, 2), _random_dirs(100, 3)
    Ya, Yb = sh.real_sh(a), sh.real_sh(b)
    t = np.sum(a * b, axis=1)
    legendre = [np.ones_like(t), t, 0.5 * (3 * t ** 2 - 1), 0.5 * (5 * t ** 3 - 3 * t)]
    for l in range(4):
        blk = slice(l * l, (l + 1) ** 2)
        lhs = np.sum(Ya[:, blk] * Yb[:, blk], axis=1)
        assert np.allclose(lhs, (2 * l + 1) / (4 * pi) * legendre[l], atol=1e-14)


def test_parity():
    """Y_lm(-n) = (-1)^l Y_lm(n)."""
    n = _random_dirs(30, 4)
    Yp, Ym = sh.real_sh(n), sh.real_sh(-n)
    for l in range(4):
        blk = slice(l * l, (l + 1) ** 2)
        assert np.allclose(Ym[:, blk], (-1) ** l * Yp[:, blk], atol=1e-15)


def test_zero_vector_defined():
    Y = sh.real_sh(np.zeros((2, 3)))
    assert np.all(np.isfinite(Y))
    assert np.allclose(Y[:, 0], 0.28209479177387814)
    assert np.all(Y[:, 1:] == 0.0)


@pytest.mark.parametrize("planted", ["drop_cs_phase", "swap_sin_cos"])
def test_pins_catch_planted_mistakes(planted, monkeypatch):
    """A plausible mistake planted in the oracle fails the scipy pin."""
    from scipy.special import sph_harm_y

    good = sh.real_sh

    def bad(vec):
        Y = good(vec).copy()
        if planted == "drop_cs_phase":
            Y[:, sh.sh_index(1, 1)] *= -1
        else:
            Y[:, [sh.sh_index(2, 1), sh.sh_index(2, -1)]] = Y[:, [sh.sh_index(2, -1), sh.sh_index(2, 1)]]
        return Y

    n = _random_dirs(20, 5)
    theta, phi = np.arccos(n[:, 2]), np.arctan2(n[:, 1], n[:, 0])
    Y = bad(n)
    ok = True
    for l in range(4):
        for m in range(1, l + 1):
            yc = sph_harm_y(l, m, theta, phi)
            ok &= np.allclose(Y[:, sh.sh_index(l, m)], sqrt(2) * yc.real, atol=1e-12)
            ok &= np.allclose(Y[:, sh.sh_index(l, -m)], sqrt(2) * yc.imag, atol=1e-12)
    assert not ok
