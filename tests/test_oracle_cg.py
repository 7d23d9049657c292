"""Pins for the oracle's Clebsch-Gordan coefficients (CPU only)."""
import json
import os
from math import factorial, pi, sqrt

import numpy as np
import pytest

from oracle import cg, sh
from tests.rotations import random_rotation, wigner_d_blocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _all_lm(lmax):
    return [(l, m) for l in range(lmax + 1) for m in range(-l, l + 1)]


def test_matches_sympy():
    sp = pytest.importorskip("sympy.physics.quantum.cg")
    for l1 in range(4):
        for l2 in range(4):
            for l3 in range(abs(l1 - l2), l1 + l2 + 1):
                for m1 in range(-l1, l1 + 1):
                    for m2 in range(-l2, l2 + 1):
                        m3 = m1 + m2
                        if abs(m3) > l3:
                            continue
                        ref = float(sp.CG(l1, m1, l2, m2, l3, m3).doit())
                        assert abs(cg.clebsch_gordan(l1, m1, l2, m2, l3, m3) - ref) < 1e-14


@pytest.mark.parametrize("l1,l2", [(1, 1), (1, 2), (2, 2), (2, 3), (3, 3)])
def test_orthogonality_relations(l1, l2):
    L3 = range(abs(l1 - l2), l1 + l2 + 1)
    rows = [(l3, m3) for l3 in L3 for m3 in range(-l3, l3 + 1)]
    cols = [(m1, m2) for m1 in range(-l1, l1 + 1) for m2 in range(-l2, l2 + 1)]
    T = np.array([[cg.clebsch_gordan(l1, m1, l2, m2, l3, m3) for (m1, m2) in cols]
                  for (l3, m3) in rows])
    # square and orthogonal: both completeness relations at once
    assert T.shape[0] == T.shape[1]
    assert np.allclose(T @ T.T, np.eye(len(rows)), atol=1e-14)
    assert np.allclose(T.T @ T, np.eye(len(cols)), atol=1e-14)


def test_special_values():
    for l in range(4):
        for m in range(-l, l + 1):
            assert abs(cg.clebsch_gordan(l, m, l, -m, 0, 0) - (-1) ** (l - m) / sqrt(2 * l + 1)) < 1e-15
            assert abs(cg.clebsch_gordan(l, m, 0, 0, l, m) - 1.0) < 1e-15
            assert abs(cg.clebsch_gordan(0, 0, l, m, l, m) - 1.0) < 1e-15
    assert cg.clebsch_gordan(1, 0, 1, 0, 1, 0) == 0.0       # odd L, all m = 0
    assert cg.clebsch_gordan(1, 1, 1, 1, 1, 1) == 0.0       # m3 != m1 + m2
    assert cg.clebsch_gordan(3, 0, 0, 0, 2, 0) == 0.0       # triangle violated


def test_path_count_is_the_pages_34():
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    ps = cg.paths()
    assert len(ps) == g["cg_entries_for_lmax3"]
    assert len(set(ps)) == len(ps)
    assert sum((l1 + l2 + l3) % 2 == 1 for l1, l2, l3 in ps) == 11
    total = sum(int(np.count_nonzero(b)) for *_, b in cg.real_cg_tables())
    assert total == 611


def test_real_tables_orthonormal():
    """For fixed (l1, l2) the real tables of all l3 stack to an orthogonal
    matrix restricted to l3 <= 3 (rows orthonormal)."""
    for l1 in range(4):
        for l2 in range(4):
            rows = []
            for (a, b, l3, blk) in cg.real_cg_tables():
                if (a, b) == (l1, l2):
                    rows.append(blk.reshape(2 * l3 + 1, -1))
            T = np.concatenate(rows, axis=0)
            assert np.allclose(T @ T.T, np.eye(T.shape[0]), atol=1e-14)


def _cg000_closed_form(l1, l2, l3):
    """<l1 0 l2 0 | l3 0> for even l1+l2+l3 (textbook closed form)."""
    L = l1 + l2 + l3
    g = L // 2
    v = sqrt((2 * l3 + 1) * factorial(L - 2 * l1) * factorial(L - 2 * l2)
             * factorial(L - 2 * l3) / factorial(L + 1))
    v *= factorial(g) / (factorial(g - l1) * factorial(g - l2) * factorial(g - l3))
    return (-1) ** (g - l3) * v


def test_even_paths_are_gaunt_integrals():
    """Even paths: C^R = Gaunt / kappa, Gaunt by sphere quadrature of SH.

    int Y_l3m3 Y_l1m1 Y_l2m2 dOmega = sqrt((2l1+1)(2l2+1)/(4pi(2l3+1)))
                                      <l1 0 l2 0|l3 0> C^R[m3, m1, m2].
    This ties the real-basis tables (values, signs, index order) to the
    harmonics themselves.
    """
    t, wt = np.polynomial.legendre.leggauss(10)
    nphi = 24
    phi = 2 * pi * np.arange(nphi) / nphi
    T, P = np.meshgrid(t, phi, indexing="ij")
    s = np.sqrt(1 - T ** 2)
    n = np.stack([s * np.cos(P), s * np.sin(P), T], axis=-1).reshape(-1, 3)
    w = (wt[:, None] * np.full(nphi, 2 * pi / nphi)[None, :]).reshape(-1)
    Y = sh.real_sh(n)
    for (l1, l2, l3, blk) in cg.real_cg_tables():
        if (l1 + l2 + l3) % 2:
            continue
        Y1 = Y[:, l1 * l1:(l1 + 1) ** 2]
        Y2 = Y[:, l2 * l2:(l2 + 1) ** 2]
        Y3 = Y[:, l3 * l3:(l3 + 1) ** 2]
        gaunt = np.einsum("q,qa,qb,qc->abc", w, Y3, Y1, Y2)
        kappa = sqrt((2 * l1 + 1) * (2 * l2 + 1) / (4 * pi * (2 * l3 + 1))) * _cg000_closed_form(l1, l2, l3)
        assert np.allclose(gaunt, kappa * blk, atol=1e-13), (l1, l2, l3)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_real_tables_intertwine_rotations(seed):
    """C^R (D_l1 (x) D_l2) = D_l3 C^R for every path, D fitted from SH."""
    D = wigner_d_blocks(random_rotation(seed))
    for (l1, l2, l3, blk) in cg.real_cg_tables():
        lhs = np.einsum("kab,ai,bj->kij", blk, D[l1], D[l2])
        rhs = np.einsum("kc,cij->kij", D[l3], blk)
        assert np.allclose(lhs, rhs, atol=1e-11), (l1, l2, l3)


def test_aligned_frame_selection_rule():
    """E2Former-V2 Eq. 13: with m2 = 0 each m3 takes at most one m1:
    m1 = +m3 on even paths, m1 = -m3 on odd paths."""
    for (l1, l2, l3, blk) in cg.real_cg_tables():
        sl = blk[:, :, l2]  # m2 = 0
        odd = (l1 + l2 + l3) % 2 == 1
        for m3 in range(-l3, l3 + 1):
            nz = [m1 for m1 in range(-l1, l1 + 1) if abs(sl[m3 + l3, m1 + l1]) > 1e-14]
            assert len(nz) <= 1
            if nz:
                assert nz[0] == (-m3 if odd else m3)


def test_planted_transpose_fails_intertwining():
    """Transposing U (a plausible slip) breaks the rotation pin."""
    D = wigner_d_blocks(random_rotation(7))
    l1, l2, l3 = 1, 2, 2
    cgc = cg.complex_cg_block(l1, l2, l3)
    u1, u2, u3 = (cg.complex_to_real(l).T for l in (l1, l2, l3))  # planted .T
    cr = np.einsum("ac,cde,bd,fe->abf", u3, cgc, u1.conj(), u2.conj())
    bad = cr.imag if np.abs(cr.imag).max() > np.abs(cr.real).max() else cr.real
    lhs = np.einsum("kab,ai,bj->kij", bad, D[l1], D[l2])
    rhs = np.einsum("kc,cij->kij", D[l3], bad)
    assert not np.allclose(lhs, rhs, atol=1e-8)
