"""Real orthonormal spherical harmonics, l <= 3, in double precision (oracle).

Definition followed
  The Batmobile blog ("Batmobile CUDA内核优化", section "2. 寄存器中间计算")
  normalises each edge vector and writes the 16 real harmonics Y_lm for
  l <= 3; it prints Y00 = 0.28209479177387814 and the l = 1 triple
  (0.4886025119029199 * z, -0.4886025119029199 * x, -0.4886025119029199 * y)
  and says l = 2, 3 are "similar". We take the textbook real orthonormal
  harmonics with the Condon-Shortley phase, which reproduce those printed
  values:

    m > 0 :  Y_lm = sqrt(2) N_lm P_l^m(z) cos(m phi)
    m < 0 :  Y_lm = sqrt(2) N_l|m| P_l^|m|(z) sin(|m| phi)
    m = 0 :  Y_l0 = N_l0 P_l(z)

  with N_lm = sqrt((2l+1)/(4 pi) (l-m)!/(l+m)!) and
  P_l^m(z) = (-1)^m (1-z^2)^(m/2) d^m/dz^m P_l(z)  (CS phase included),
  P_l from Rodrigues' formula.  On the unit sphere
  (1-z^2)^(m/2) e^(i m phi) = (x + i y)^m, so everything is a polynomial in
  the unit vector (x, y, z).

Layout: component index k = l*l + l + m, m = -l..l (16 components for
l <= 3; (l_max+1)^2 in general).

Zero-length vectors (not produced by the graph generator) are given n = 0,
so Y_00 is the constant and every l >= 1 component is 0: defined, never NaN.
"""
from math import factorial, pi, sqrt

import numpy as np
from numpy.polynomial import Polynomial

L_MAX = 3
N_SH = (L_MAX + 1) ** 2  # 16


def sh_index(l: int, m: int) -> int:
    """Position of (l, m) in the 16-vector."""
    return l * l + l + m


def legendre_polynomial(l: int) -> Polynomial:
    """P_l by Rodrigues' formula: P_l = 1/(2^l l!) d^l/dz^l (z^2 - 1)^l."""
    base = Polynomial([-1.0, 0.0, 1.0]) ** l
    return base.deriv(l) / (2.0 ** l * factorial(l))


def normalisation(l: int, m: int) -> float:
    """N_lm = sqrt((2l+1)/(4 pi) * (l-m)!/(l+m)!), m >= 0."""
    return sqrt((2 * l + 1) / (4.0 * pi) * factorial(l - m) / factorial(l + m))


def unit_vectors(vec: np.ndarray) -> np.ndarray:
    """n = v/|v| row by row; rows with |v|^2 < 1e-30 map to n = 0."""
    vec = np.asarray(vec, dtype=np.float64).reshape(-1, 3)
    r2 = np.einsum("ij,ij->i", vec, vec)
    out = np.zeros_like(vec)
    ok = r2 >= 1e-30
    out[ok] = vec[ok] / np.sqrt(r2[ok])[:, None]
    return out


def real_sh(vec: np.ndarray, l_max: int = L_MAX) -> np.ndarray:
    """Y[E, (l_max+1)^2] for edge vectors vec[E, 3] (need not be unit length).

    The same definition for every degree; l_max = 3 (16 components) is the
    Batmobile layer, larger l_max the higher-degree variant that the blog
    names as its limitation (section on limits and future work).
    """
    n = unit_vectors(vec)
    x, y, z = n[:, 0], n[:, 1], n[:, 2]
    xy = x + 1j * y
    out = np.zeros((n.shape[0], (l_max + 1) ** 2), dtype=np.float64)
    for l in range(l_max + 1):
        pl = legendre_polynomial(l)
        for m in range(0, l + 1):
            # P_l^m(z) (1-z^2)^(-m/2) = (-1)^m d^m P_l / dz^m
            dpl = pl.deriv(m) if m > 0 else pl
            radial = (-1.0) ** m * dpl(z)
            if m == 0:
                out[:, sh_index(l, 0)] = normalisation(l, 0) * radial
            else:
                pw = xy ** m  # (x + i y)^m = (1-z^2)^(m/2) e^(i m phi)
                c = sqrt(2.0) * normalisation(l, m) * radial
                out[:, sh_index(l, m)] = c * pw.real
                out[:, sh_index(l, -m)] = c * pw.imag
    # n = 0 rows: the l >= 1 polynomials above vanish at the origin except
    # the constant parts of P_l(z) (e.g. -1/2 in P_2); force them to 0.
    zero = ~np.any(n != 0.0, axis=1)
    out[zero, 1:] = 0.0
    return out
