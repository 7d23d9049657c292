"""Build-time generator of the constexpr tables used by the CUDA kernels.

Writes ``eqmp_tables.h``: the 34 real-basis Clebsch-Gordan paths for
l <= 3 (every triangle-allowed (l1, l2, l3), parity unrestricted, in the
order l1 = 0..3, l2 = 0..3, l3 = |l1-l2|..min(3, l1+l2)), their nonzero
terms (k3, k1, k2, value) with k = l*l + l + m, and the real spherical
harmonic normalisation constants.  The Batmobile blog ("Batmobile
CUDA内核优化", section "1. 编译时常量") bakes the CG coefficients into the
kernel as compile-time constants so that the compiler can fold them into
the instruction stream; this file produces those constants.

Method (independent of any other implementation in this repository):
  * Wigner 3j symbols from Racah's single-sum formula, evaluated exactly
    (squared magnitude as a Fraction, sign tracked separately);
  * complex CG  <l1 m1 l2 m2 | l3 m3> = (-1)^(l1-l2+m3) sqrt(2 l3 + 1)
    (l1 l2 l3; m1 m2 -m3);
  * real basis: real Y_l = U_l complex Y_l with, for m > 0,
    row m = (Y^m + (-1)^m Y^-m)/sqrt2 and row -m = i ((-1)^m Y^-m - Y^m)/sqrt2,
    row 0 = Y^0; the real tensor is U3 CG (U1 (x) U2)^H.  It is real for
    even l1+l2+l3 and imaginary for odd; the odd ones are multiplied by -i.

Run:  python gen_tables.py OUT_HEADER
"""
import sys
from fractions import Fraction
from math import factorial, pi, sqrt

LMAX = 3


def _fact(n):
    return factorial(n)


def wigner_3j(j1, j2, j3, m1, m2, m3):
    """(j1 j2 j3; m1 m2 m3) as a float (Racah single sum, exact inside)."""
    if m1 + m2 + m3 != 0 or not (abs(j1 - j2) <= j3 <= j1 + j2):
        return 0.0
    if abs(m1) > j1 or abs(m2) > j2 or abs(m3) > j3:
        return 0.0
    tri = Fraction(_fact(j1 + j2 - j3) * _fact(j1 - j2 + j3) * _fact(-j1 + j2 + j3),
                   _fact(j1 + j2 + j3 + 1))
    mag2 = tri * (_fact(j1 + m1) * _fact(j1 - m1) * _fact(j2 + m2) * _fact(j2 - m2)
                  * _fact(j3 + m3) * _fact(j3 - m3))
    s = Fraction(0)
    kmin = max(0, j2 - j3 - m1, j1 - j3 + m2)
    kmax = min(j1 + j2 - j3, j1 - m1, j2 + m2)
    for k in range(kmin, kmax + 1):
        s += Fraction((-1) ** k, _fact(k) * _fact(j1 + j2 - j3 - k) * _fact(j1 - m1 - k)
                      * _fact(j2 + m2 - k) * _fact(j3 - j2 + m1 + k) * _fact(j3 - j1 - m2 + k))
    if s == 0:
        return 0.0
    sign = (-1) ** (j1 - j2 - m3)
    sign = sign if s > 0 else -sign
    return sign * sqrt(float(mag2 * s * s))


def cg_complex(l1, m1, l2, m2, l3, m3):
    if m1 + m2 != m3:
        return 0.0
    return (-1) ** (l1 - l2 + m3) * sqrt(2 * l3 + 1) * wigner_3j(l1, l2, l3, m1, m2, -m3)


def u_row(l, m):
    """Row m of U_l as {mu: complex coefficient}."""
    r = 1.0 / sqrt(2.0)
    if m == 0:
        return {0: 1.0 + 0j}
    a = abs(m)
    sgn = (-1) ** a
    if m > 0:
        return {a: r + 0j, -a: sgn * r + 0j}
    return {-a: 1j * sgn * r, a: -1j * r}


def real_cg(l1, l2, l3):
    """{(m3, m1, m2): value} nonzero real-basis entries of one path."""
    odd = (l1 + l2 + l3) % 2 == 1
    out = {}
    for m3 in range(-l3, l3 + 1):
        for m1 in range(-l1, l1 + 1):
            for m2 in range(-l2, l2 + 1):
                acc = 0j
                for mu3, a3 in u_row(l3, m3).items():
                    for mu1, a1 in u_row(l1, m1).items():
                        for mu2, a2 in u_row(l2, m2).items():
                            c = cg_complex(l1, mu1, l2, mu2, l3, mu3)
                            if c:
                                acc += a3 * c * a1.conjugate() * a2.conjugate()
                v = (-1j * acc) if odd else acc
                if abs(v.imag) > 1e-12:
                    raise RuntimeError(f"path {(l1, l2, l3)} not reducible to a real table")
                if abs(v.real) > 1e-13:
                    out[(m3, m1, m2)] = v.real
    return out


def all_paths(lmax=LMAX):
    return [(a, b, c) for a in range(lmax + 1) for b in range(lmax + 1)
            for c in range(abs(a - b), min(lmax, a + b) + 1)]


def k_of(l, m):
    return l * l + l + m


def sh_constants():
    """Real SH as K_lm * Q_lm(z) * {Re, Im}(x + i y)^|m| on the unit sphere.

    Q_lm(z) = (-1)^m d^m/dz^m P_l(z) (Condon-Shortley phase), coefficients
    in ascending powers of z; K_lm = sqrt2 N_lm (m > 0) or N_l0, with
    N_lm = sqrt((2l+1)/(4pi) (l-m)!/(l+m)!).  Returns {(l, m>=0): [c0, c1, ...]}
    with K folded into the coefficients.
    """
    # Legendre P_l coefficients (ascending powers), exact.
    P = {0: [Fraction(1)], 1: [Fraction(0), Fraction(1)],
         2: [Fraction(-1, 2), Fraction(0), Fraction(3, 2)],
         3: [Fraction(0), Fraction(-3, 2), Fraction(0), Fraction(5, 2)]}
    out = {}
    for l in range(LMAX + 1):
        for m in range(0, l + 1):
            c = list(P[l])
            for _ in range(m):
                c = [c[i] * i for i in range(1, len(c))] or [Fraction(0)]
            c = [(-1) ** m * v for v in c]
            norm = sqrt((2 * l + 1) / (4 * pi) * _fact(l - m) / _fact(l + m))
            K = norm * (sqrt(2.0) if m > 0 else 1.0)
            out[(l, m)] = [float(v) * K for v in c]
    return out


def _f(v):
    t = f"{v:.17g}"
    if "." not in t and "e" not in t and "inf" not in t and "nan" not in t:
        t += ".0"
    return t + "f"


def render():
    paths = all_paths()
    lines = []
    terms = []
    first = []
    for (l1, l2, l3) in paths:
        ent = real_cg(l1, l2, l3)
        first.append(len(terms))
        for (m3, m1, m2) in sorted(ent):
            terms.append((k_of(l3, m3), k_of(l1, m1), k_of(l2, m2), ent[(m3, m1, m2)]))
    lines += [
        "// Generated by gen_tables.py at build time. Do not edit.",
        "#pragma once",
        "namespace eqmp { namespace tables {",
        f"constexpr int kNumPaths = {len(paths)};",
        f"constexpr int kNumTerms = {len(terms)};",
        "struct Path { int l1, l2, l3, first, count; };",
        "struct Term { int k3, k1, k2; float c; };",
        "constexpr Path kPaths[kNumPaths] = {",
    ]
    for i, (l1, l2, l3) in enumerate(paths):
        nxt = first[i + 1] if i + 1 < len(paths) else len(terms)
        lines.append(f"  {{{l1}, {l2}, {l3}, {first[i]}, {nxt - first[i]}}},")
    lines.append("};")
    lines.append("// terms grouped by path, then (m3, m1, m2) ascending")
    lines.append("constexpr Term kTerms[kNumTerms] = {")
    for (k3, k1, k2, v) in terms:
        lines.append(f"  {{{k3}, {k1}, {k2}, {_f(v)}}},")
    lines.append("};")
    shc = sh_constants()
    lines.append("// real SH: Y_lm = poly_lm(z) * {Re,Im}(x+iy)^|m|, poly coefficients ascending in z")
    lines.append("constexpr float kShPoly[4][4][4] = {  // [l][|m|][power]")
    for l in range(LMAX + 1):
        row = []
        for m in range(LMAX + 1):
            c = shc.get((l, m), [])
            c = (c + [0.0] * 4)[:4]
            row.append("{" + ", ".join(_f(v) for v in c) + "}")
        lines.append("  {" + ", ".join(row) + "},")
    lines.append("};")
    # aligned-frame (SO(2)) tables
    at = aligned_terms()
    lines.append("// aligned frame: m'[k3] += W_p * kappa * x'[k1]  (E2Former-V2 Eq. 13 form)")
    lines.append("struct AlignedTerm { int p, k3, k1; float kappa; };")
    lines.append(f"constexpr int kNumAligned = {len(at)};")
    lines.append("constexpr AlignedTerm kAligned[kNumAligned] = {")
    for (pp, k3, k1, kap) in at:
        lines.append(f"  {{{pp}, {k3}, {k1}, {_f(kap)}}},")
    lines.append("};")
    ir = ir_coefficients()
    for nm, idx in (("kIrU", 0), ("kIrV", 1), ("kIrW", 2)):
        lines.append(f"constexpr float {nm}[2][7][7] = {{  // [l-2][m+3][n+3] (zero outside |m|,|n| <= l)")
        for l in (2, 3):
            rows = []
            for m in range(-3, 4):
                vals = []
                for n in range(-3, 4):
                    vals.append(_f(ir[l][m + l][n + l][idx]) if abs(m) <= l and abs(n) <= l else "0.0f")
                rows.append("{" + ", ".join(vals) + "}")
            lines.append("  {" + ", ".join(rows) + "},")
        lines.append("};")
    lines.append("}}  // namespace eqmp::tables")
    return "\n".join(lines) + "\n", paths, terms


def main(argv):
    text, paths, terms = render()
    if len(argv) > 1:
        with open(argv[1], "w") as fh:
            fh.write(text)
    else:
        sys.stdout.write(text)



# ---------------------------------------------------------------------------
# Aligned-frame (SO(2)) form of the same tensor product, E2Former-V2 section
# 2.1 (EAAS): rotate x into a frame whose z axis is the edge, where the edge
# harmonics keep only m = 0 (Lemma 4.1) and each output m3 takes at most one
# input m1 (Eq. 13); rotate the result back.  Everything below is computed
# here independently and emitted as constexpr tables.

def aligned_terms(lmax=LMAX):
    """[(p, k3, k1, kappa)]: m'[k3] += W_p kappa x'[k1] in the edge frame.

    kappa = C_p[m3, m1, m2=0] * Y_l2,0(z-axis), Y_l,0(z) = sqrt((2l+1)/(4 pi)).
    """
    out = []
    for p, (l1, l2, l3) in enumerate(all_paths(lmax)):
        ent = real_cg(l1, l2, l3)
        yz = sqrt((2 * l2 + 1) / (4 * pi))
        for (m3, m1, m2), v in sorted(ent.items()):
            if m2 == 0:
                out.append((p, k_of(l3, m3), k_of(l1, m1), v * yz))
    return out


def frame_from_direction(n):
    """Right-handed orthonormal (t1, t2, n) with n the unit edge direction
    (branch-free construction of an orthonormal basis from one vector,
    Duff et al. 2017).  Returns the 3x3 rotation Q with columns t1, t2, n."""
    x, y, z = n
    s = 1.0 if z >= 0.0 else -1.0
    a = -1.0 / (s + z)
    b = x * y * a
    t1 = (1.0 + s * x * x * a, s * b, -s * x)
    t2 = (b, s + y * y * a, -y)
    return [[t1[0], t2[0], x], [t1[1], t2[1], y], [t1[2], t2[2], z]]


def ir_coefficients(levels=(2, 3)):
    """Ivanic-Ruedenberg recursion coefficients u, v, w for the given l:
    {l: [[(u, v, w) for n in -l..l] for m in -l..l]}."""
    out = {}
    for l in levels:
        rows = []
        for m in range(-l, l + 1):
            row = []
            for n in range(-l, l + 1):
                d = 1 if m == 0 else 0
                den = (2 * l) * (2 * l - 1) if abs(n) == l else (l + n) * (l - n)
                u = sqrt((l + m) * (l - m) / den)
                v = 0.5 * sqrt((1 + d) * (l + abs(m) - 1) * (l + abs(m)) / den) * (1 - 2 * d)
                w = -0.5 * sqrt((l - abs(m) - 1) * (l - abs(m)) / den) * (1 - d)
                row.append((u, v, w))
            rows.append(row)
        out[l] = rows
    return out


def wigner_real(Q, lmax=3):
    """Real Wigner-D blocks D_1..D_lmax in this library's SH basis (CS phase,
    k = l*l+l+m) for rotation Q: Y_l(Q v) = D_l Y_l(v).  Plain Python
    reference of the device recursion."""
    # l = 1 in the (y, z, x) ordering without signs
    idx = [1, 2, 0]
    R = [[Q[idx[i]][idx[j]] for j in range(3)] for i in range(3)]
    D = {1: R}
    coef = ir_coefficients(tuple(range(2, lmax + 1)))

    def Rm(i, j):
        return R[i + 1][j + 1]

    def Dl(l, a, b):
        return D[l][a + l][b + l]

    def P(i, l, a, b):
        if b == l:
            return Rm(i, 1) * Dl(l - 1, a, l - 1) - Rm(i, -1) * Dl(l - 1, a, -l + 1)
        if b == -l:
            return Rm(i, 1) * Dl(l - 1, a, -l + 1) + Rm(i, -1) * Dl(l - 1, a, l - 1)
        return Rm(i, 0) * Dl(l - 1, a, b)

    for l in range(2, lmax + 1):
        M = []
        for m in range(-l, l + 1):
            row = []
            for n in range(-l, l + 1):
                u, v, w = coef[l][m + l][n + l]
                val = 0.0
                if u != 0.0:
                    val += u * P(0, l, m, n)
                if v != 0.0:
                    if m == 0:
                        V = P(1, l, 1, n) + P(-1, l, -1, n)
                    elif m > 0:
                        V = P(1, l, m - 1, n) * sqrt(1 + (m == 1)) - P(-1, l, -m + 1, n) * (1 - (m == 1))
                    else:
                        V = P(1, l, m + 1, n) * (1 - (m == -1)) + P(-1, l, -m - 1, n) * sqrt(1 + (m == -1))
                    val += v * V
                if w != 0.0:
                    if m > 0:
                        W = P(1, l, m + 1, n) + P(-1, l, -m - 1, n)
                    else:
                        W = P(1, l, m - 1, n) - P(-1, l, -m + 1, n)
                    val += w * W
                row.append(val)
            M.append(row)
        D[l] = M
    # this library's basis carries the Condon-Shortley sign (-1)^|m| on m != 0
    out = {}
    for l in range(1, lmax + 1):
        sg = [(-1) ** abs(m) if m != 0 else 1 for m in range(-l, l + 1)]
        out[l] = [[sg[i] * D[l][i][j] * sg[j] for j in range(2 * l + 1)] for i in range(2 * l + 1)]
    return out


# ---------------------------------------------------------------------------
# Higher degrees (l_max = 4..6), the aligned-frame schedule only: the blog
# names l <= 3 as its limit; at higher degree the dense product grows as
# l^6 terms while the aligned one grows as l^3 (E2Former-V2 sections 1.1 and
# 2.1), so only the aligned tables are emitted.

HIGH_DEGREES = (4, 5, 6)


def render_high():
    lines = [
        "// Generated by gen_tables.py at build time. Do not edit.",
        "#pragma once",
        "#include <cuda_runtime.h>",
        "namespace eqmp { namespace tables_hl {",
        "struct HlPath { int l1, l2, l3, first, count; };",
        "struct HlTerm { int k3, k1; float kappa; };",
        "template <int L> struct Hl;",
    ]
    for L in HIGH_DEGREES:
        paths = all_paths(L)
        at = aligned_terms(L)
        first, count = [], []
        for p in range(len(paths)):
            idx = [i for i, t in enumerate(at) if t[0] == p]
            first.append(idx[0] if idx else len(at))
            count.append(len(idx))
        lines.append(f"template <> struct Hl<{L}> {{")
        lines.append(f"  static constexpr int kNumPaths = {len(paths)};")
        lines.append(f"  static constexpr int kNumTerms = {len(at)};")
        lines.append(f"  static constexpr HlPath kPaths[{len(paths)}] = {{")
        for p, (l1, l2, l3) in enumerate(paths):
            lines.append(f"    {{{l1}, {l2}, {l3}, {first[p]}, {count[p]}}},")
        lines.append("  };")
        lines.append(f"  static constexpr HlTerm kTerms[{len(at)}] = {{")
        for (pp, k3, k1, kap) in at:
            lines.append(f"    {{{k3}, {k1}, {_f(kap)}}},")
        lines.append("  };")
        lines.append("};")
    top = max(HIGH_DEGREES)
    ir = ir_coefficients(tuple(range(2, top + 1)))
    W = 2 * top + 1
    for nm, idx in (("kHlIrU", 0), ("kHlIrV", 1), ("kHlIrW", 2)):
        lines.append(f"// Ivanic-Ruedenberg {nm[-1].lower()} for l = 2..{top}: [l-2][m+{top}][n+{top}] (0 outside |m|,|n| <= l)")
        lines.append(f"constexpr float {nm}[{top - 1}][{W}][{W}] = {{")
        for l in range(2, top + 1):
            rows = []
            for m in range(-top, top + 1):
                vals = []
                for n in range(-top, top + 1):
                    vals.append(_f(ir[l][m + l][n + l][idx]) if abs(m) <= l and abs(n) <= l else "0.0f")
                rows.append("{" + ", ".join(vals) + "}")
            lines.append("  {" + ", ".join(rows) + "},")
        lines.append("};")
    lines.append("}}  // namespace eqmp::tables_hl")
    return "\n".join(lines) + "\n"


if __name__ == "__main__":
    if len(sys.argv) > 2 and sys.argv[1] == "--high":
        with open(sys.argv[2], "w") as fh:
            fh.write(render_high())
    else:
        main(sys.argv)
