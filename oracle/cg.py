"""Clebsch-Gordan coefficients, complex and real basis (oracle).

Paths
  The Batmobile blog ("Batmobile CUDA内核优化", section "1. 编译时常量")
  bakes 34 CG entries for L_MAX = 3 into the kernel.  34 is the number of
  triangle-allowed triples (l1, l2, l3) with every l <= 3 and no parity
  filter, so every such path is taken, including the odd ones
  (l1 + l2 + l3 odd).  Order: l1 = 0..3, l2 = 0..3, l3 = |l1-l2|..min(3, l1+l2).

Complex CG
  <l1 m1 l2 m2 | l3 m3> by Racah's closed formula (Condon-Shortley
  convention, unit-normalised CG, not the 3j symbol), evaluated with exact
  integers and one final square root.

Real basis
  With U_l the unitary taking complex SH to the real SH of ``oracle.sh``
  (rows: m > 0 -> (Y^m + (-1)^m Y^-m)/sqrt2, m < 0 -> -i (Y^|m| -
  (-1)^|m| Y^-|m|)/sqrt2, m = 0 -> Y^0):

      C^R[m3, m1, m2] = sum U3[m3, u3] CG[u3; u1, u2] conj(U1[m1, u1]) conj(U2[m2, u2])

  which is purely real for even l1+l2+l3 and purely imaginary for odd.
  Reading taken: real part for even paths, imaginary part for odd paths
  (the pages fix no sign for the odd, pseudo-tensor paths; any per-path
  sign is absorbed by its weight).  E2Former-V2 (section 2.1, Eq. 13)
  states the structure this must have: in a frame where the edge lies on
  z only m2 = 0 survives, and each output m3 then comes from at most one
  input m1 (m3 = +m1 for even, m3 = -m1 for odd paths).
"""
from fractions import Fraction
from functools import lru_cache
from math import factorial, sqrt

import numpy as np

L_MAX = 3


def paths(l_max: int = L_MAX):
    """The triangle-allowed (l1, l2, l3), all <= l_max, lexicographic
    (34 for l_max = 3)."""
    out = []
    for l1 in range(l_max + 1):
        for l2 in range(l_max + 1):
            for l3 in range(abs(l1 - l2), min(l_max, l1 + l2) + 1):
                out.append((l1, l2, l3))
    return out


def clebsch_gordan(l1, m1, l2, m2, l3, m3) -> float:
    """<l1 m1 l2 m2 | l3 m3>, Racah's formula."""
    if m1 + m2 != m3:
        return 0.0
    if not (abs(l1 - l2) <= l3 <= l1 + l2):
        return 0.0
    if abs(m1) > l1 or abs(m2) > l2 or abs(m3) > l3:
        return 0.0
    f = factorial
    # squared prefactor, exact
    pref = Fraction(
        (2 * l3 + 1) * f(l3 + l1 - l2) * f(l3 - l1 + l2) * f(l1 + l2 - l3),
        f(l1 + l2 + l3 + 1),
    )
    pref *= (f(l3 + m3) * f(l3 - m3) * f(l1 - m1) * f(l1 + m1)
             * f(l2 - m2) * f(l2 + m2))
    total = Fraction(0)
    for k in range(0, l1 + l2 - l3 + 1):
        d = [k, l1 + l2 - l3 - k, l1 - m1 - k, l2 + m2 - k,
             l3 - l2 + m1 + k, l3 - l1 - m2 + k]
        if min(d) < 0:
            continue
        den = 1
        for v in d:
            den *= f(v)
        total += Fraction((-1) ** k, den)
    if total == 0:
        return 0.0
    sign = 1.0 if total > 0 else -1.0
    return sign * sqrt(float(pref * total * total))


def complex_to_real(l: int) -> np.ndarray:
    """U_l, (2l+1)x(2l+1): real Y_l = U_l @ complex Y_l; index m + l."""
    u = np.zeros((2 * l + 1, 2 * l + 1), dtype=np.complex128)
    s = 1.0 / sqrt(2.0)
    for m in range(-l, l + 1):
        r = m + l
        if m == 0:
            u[r, l] = 1.0
        elif m > 0:
            u[r, l + m] = s
            u[r, l - m] = (-1) ** m * s
        else:
            a = -m
            u[r, l + a] = -1j * s
            u[r, l - a] = 1j * (-1) ** a * s
    return u


def complex_cg_block(l1, l2, l3) -> np.ndarray:
    """CG[u3 + l3, u1 + l1, u2 + l2] for one path."""
    t = np.zeros((2 * l3 + 1, 2 * l1 + 1, 2 * l2 + 1))
    for u1 in range(-l1, l1 + 1):
        for u2 in range(-l2, l2 + 1):
            u3 = u1 + u2
            if abs(u3) <= l3:
                t[u3 + l3, u1 + l1, u2 + l2] = clebsch_gordan(l1, u1, l2, u2, l3, u3)
    return t


@lru_cache(maxsize=None)
def real_cg_block(l1, l2, l3) -> np.ndarray:
    """C^R[m3 + l3, m1 + l1, m2 + l2] (real) for one path."""
    cg = complex_cg_block(l1, l2, l3)
    u1, u2, u3 = complex_to_real(l1), complex_to_real(l2), complex_to_real(l3)
    cr = np.einsum("ac,cde,bd,fe->abf", u3, cg, u1.conj(), u2.conj())
    if (l1 + l2 + l3) % 2 == 0:
        part, other = cr.real, cr.imag
    else:
        part, other = cr.imag, cr.real
    if np.max(np.abs(other)) > 1e-12:
        raise AssertionError(f"real-basis CG of path {(l1, l2, l3)} is not pure")
    out = np.where(np.abs(part) < 1e-14, 0.0, part)
    out.setflags(write=False)
    return out


def real_cg_tables(l_max: int = L_MAX):
    """[(l1, l2, l3, C^R block)] for all paths (34 for l_max = 3) in order."""
    return [(l1, l2, l3, real_cg_block(l1, l2, l3)) for (l1, l2, l3) in paths(l_max)]
