"""Pins for the oracle at degrees above 3 (l_max = 4..6), CPU only.

The Batmobile blog names l <= 3 as its limit and higher degrees as future
work; the oracle's definitions are written for any degree, and these tests
fix them there by things other than the oracle itself: scipy's complex
harmonics (library routine), exact quadrature, the addition theorem, the
aligned-frame property of the harmonics (E2Former-V2 Lemma 4.1), sympy's
CG coefficients (library routine), CG orthogonality, brute force from the
formula, rotation equivariance and the consistency of degrees (the l <= 3
part of a higher-degree layer is the l <= 3 layer).
"""
import itertools
from math import pi, sqrt

import numpy as np
import pytest

from oracle import cg, layer, sh
from tests.rotations import random_rotation, rotate_features, wigner_d_blocks

L_HIGH = (4, 5, 6)


def _dirs(n, seed):
    v = np.random.default_rng(seed).standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


@pytest.mark.parametrize("l_max", L_HIGH)
def test_sh_matches_scipy(l_max):
    from scipy.special import sph_harm_y

    n = _dirs(150, l_max)
    theta = np.arccos(np.clip(n[:, 2], -1, 1))
    phi = np.arctan2(n[:, 1], n[:, 0])
    Y = sh.real_sh(n, l_max)
    assert Y.shape == (150, (l_max + 1) ** 2)
    for l in range(l_max + 1):
        for m in range(-l, l + 1):
            yc = sph_harm_y(l, abs(m), theta, phi)
            ref = yc.real if m == 0 else (sqrt(2.0) * yc.real if m > 0 else sqrt(2.0) * yc.imag)
            assert np.allclose(Y[:, sh.sh_index(l, m)], ref, rtol=0, atol=1e-12), (l, m)


@pytest.mark.parametrize("l_max", L_HIGH)
def test_sh_orthonormal_by_quadrature(l_max):
    """Gauss-Legendre in cos(theta) x uniform phi, exact for degree <= 2 l_max."""
    t, wt = np.polynomial.legendre.leggauss(l_max + 2)
    nphi = 2 * l_max + 3
    phi = 2 * pi * np.arange(nphi) / nphi
    T, P = np.meshgrid(t, phi, indexing="ij")
    s = np.sqrt(1 - T ** 2)
    n = np.stack([s * np.cos(P), s * np.sin(P), T], axis=-1).reshape(-1, 3)
    w = (wt[:, None] * np.full(nphi, 2 * pi / nphi)[None, :]).reshape(-1)
    Y = sh.real_sh(n, l_max)
    gram = Y.T @ (Y * w[:, None])
    assert np.allclose(gram, np.eye((l_max + 1) ** 2), atol=1e-12)


@pytest.mark.parametrize("l_max", L_HIGH)
def test_addition_theorem_and_z_axis(l_max):
    Y = sh.real_sh(_dirs(50, 3), l_max)
    for l in range(l_max + 1):
        blk = slice(l * l, (l + 1) ** 2)
        assert np.allclose(np.sum(Y[:, blk] ** 2, axis=1), (2 * l + 1) / (4 * pi), atol=1e-12)
    z = sh.real_sh(np.array([[0.0, 0.0, 2.5]]), l_max)[0]
    for l in range(l_max + 1):
        for m in range(-l, l + 1):
            want = sqrt((2 * l + 1) / (4 * pi)) if m == 0 else 0.0
            assert abs(z[sh.sh_index(l, m)] - want) < 1e-12


def test_cg_matches_sympy_at_high_degree():
    from sympy import S
    from sympy.physics.quantum.cg import CG

    rng = np.random.default_rng(0)
    for _ in range(40):
        l1, l2 = (int(v) for v in rng.integers(0, 7, 2))
        l3 = int(rng.integers(abs(l1 - l2), min(6, l1 + l2) + 1))
        m1 = int(rng.integers(-l1, l1 + 1))
        m2 = int(rng.integers(-l2, l2 + 1))
        if abs(m1 + m2) > l3:
            continue
        want = float(CG(S(l1), S(m1), S(l2), S(m2), S(l3), S(m1 + m2)).doit())
        assert abs(cg.clebsch_gordan(l1, m1, l2, m2, l3, m1 + m2) - want) < 1e-12


@pytest.mark.parametrize("l_max", L_HIGH)
def test_real_cg_counts_and_orthogonality(l_max):
    tabs = cg.real_cg_tables(l_max)
    n_paths = {4: 65, 5: 111, 6: 175}[l_max]
    assert len(tabs) == n_paths == len(cg.paths(l_max))
    for l1, l2, l3, blk in tabs:
        # rows (m3) of a real CG block are orthonormal over (m1, m2)
        flat = blk.reshape(2 * l3 + 1, -1)
        assert np.allclose(flat @ flat.T, np.eye(2 * l3 + 1), atol=1e-12)
    # the first 34 paths of any degree are the l <= 3 paths
    assert [t[:3] for t in tabs if max(t[:3]) <= 3] == cg.paths(3)


def _graph(seed, n=3, C=2, l_max=4):
    rng = np.random.default_rng(seed)
    pos = rng.uniform(-2, 2, (n, 3))
    pairs = [(i, j) for i in range(n) for j in range(n) if i != j]
    dst = np.array([p[0] for p in pairs])
    src = np.array([p[1] for p in pairs])
    off = np.searchsorted(dst, np.arange(n + 1))
    P = len(cg.paths(l_max))
    x = rng.standard_normal((n, C, (l_max + 1) ** 2))
    w = rng.standard_normal((P, C))
    R = rng.standard_normal((len(src), 8))
    M = rng.standard_normal((8, P * C))
    return pos[src] - pos[dst], src, dst, off, x, w, R, M


@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_brute_force_at_degree_four(mode):
    l_max = 4
    vec, src, dst, off, x, w, R, M = _graph(1, l_max=l_max)
    kw = dict(w=w) if mode == "shared" else dict(R=R, M=M)
    got = layer.message_pass(vec, x, off, src, **kw)
    C = x.shape[1]
    want = np.zeros_like(got)
    for e in range(len(src)):
        Y = sh.real_sh(vec[e:e + 1], l_max)[0]
        for p, (l1, l2, l3, blk) in enumerate(cg.real_cg_tables(l_max)):
            for c in range(C):
                W = w[p, c] if mode == "shared" else sum(R[e, k] * M[k, p * C + c] for k in range(8))
                for m3, m1, m2 in itertools.product(range(-l3, l3 + 1), range(-l1, l1 + 1), range(-l2, l2 + 1)):
                    coef = blk[m3 + l3, m1 + l1, m2 + l2]
                    if coef:
                        want[dst[e], c, sh.sh_index(l3, m3)] += (
                            W * coef * x[src[e], c, sh.sh_index(l1, m1)] * Y[sh.sh_index(l2, m2)])
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("l_max", (4, 6))
def test_rotation_equivariance_high_degree(l_max):
    vec, src, dst, off, x, w, R, M = _graph(2, n=5, C=2, l_max=l_max)
    Q = random_rotation(9)
    D = wigner_d_blocks(Q, l_max=l_max)
    base = layer.message_pass(vec, x, off, src, w=w)
    rot = layer.message_pass(vec @ Q.T, rotate_features(x, D), off, src, w=w)
    assert np.max(np.abs(rot - rotate_features(base, D))) < 1e-10 * max(1.0, np.max(np.abs(base)))


def test_low_degree_part_is_the_l3_layer():
    """With x and the weights confined to l <= 3, the l <= 3 outputs of the
    degree-5 layer are the degree-3 layer's outputs."""
    l_max = 5
    vec, src, dst, off, x, w, R, M = _graph(3, n=4, C=3, l_max=l_max)
    x[:, :, 16:] = 0.0
    low = [i for i, p in enumerate(cg.paths(l_max)) if max(p) <= 3]
    w5 = np.zeros_like(w)
    w5[low] = w[low]
    hi = layer.message_pass(vec, x, off, src, w=w5)
    lo = layer.message_pass(vec, x[:, :, :16], off, src, w=w[low])
    assert np.allclose(hi[:, :, :16], lo, atol=1e-12)


def test_scalar_features_high_degree():
    """x only in l1 = 0: out[(l, m)] = sum_e w[(0, l, l)] x0 Y_e[(l, m)]."""
    l_max = 6
    vec, src, dst, off, x, w, R, M = _graph(4, n=3, C=2, l_max=l_max)
    x[:, :, 1:] = 0.0
    got = layer.message_pass(vec, x, off, src, w=w)
    Y = sh.real_sh(vec, l_max)
    pidx = {p: i for i, p in enumerate(cg.paths(l_max))}
    want = np.zeros_like(got)
    for e in range(len(src)):
        for l in range(l_max + 1):
            blk = slice(l * l, (l + 1) ** 2)
            want[dst[e], :, blk] += w[pidx[(0, l, l)]][:, None] * x[src[e], :, 0][:, None] * Y[e, blk][None, :]
    assert np.allclose(got, want, atol=1e-12)
