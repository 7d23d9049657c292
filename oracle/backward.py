"""Gradients of the fused layer (oracle, float64; test infrastructure).

The forward map is the one in ``oracle.layer``:
  out[i,c,k3] = sum_{e->i} sum_p W[e,p,c] sum_{k1,k2} C_p[k3,k1,k2] x[src_e,c,k1] Y(vec_e)[k2]
Given an upstream gradient g = dL/dout, this module writes the chain rule
out plainly, one factor at a time:

  dL/dx[j,c,k1]   = sum_{e: src_e=j} sum_p W[e,p,c] sum_{k3,k2} C_p[k3,k1,k2] g[dst_e,c,k3] Y_e[k2]
  s[e,p,c]        = sum_{k3,k1,k2} C_p[k3,k1,k2] g[dst_e,c,k3] x[src_e,c,k1] Y_e[k2]
  dL/dw[p,c]      = sum_e s[e,p,c]                          (shared weights)
  dL/dR[e,k]      = sum_{p,c} M[k,p*C+c] s[e,p,c]           (radial weights)
  dL/dM[k,p*C+c]  = sum_e R[e,k] s[e,p,c]
  dY[e,k2]        = sum_c sum_p W[e,p,c] sum_{k3,k1} C_p[k3,k1,k2] g[dst_e,c,k3] x[src_e,c,k1]
  dL/dvec[e]      = dY[e,:] . dY(vec_e)/dvec_e              (forces through the harmonics)

The derivative of the harmonics follows the polynomial form of
``oracle.sh`` (Y_lm = K_lm Q_lm(z) {Re,Im}(x+iy)^|m| on the unit sphere, n =
v/|v|): dY/dv = J(n) (I - n n^T) / |v|, with J the Jacobian of the
polynomial in (x, y, z).  Pinned by central finite differences of the
forward oracle (tests/test_oracle_backward.py).  For zero-length vectors
the gradient is taken as 0 (Y is constant there by the stated reading).
"""
from math import factorial, sqrt

import numpy as np

from . import cg as _cg
from . import sh as _sh

N_SH = 16


def _block(l):
    return slice(l * l, (l + 1) * (l + 1))


def _weights(p, C, edges, w, R, M):
    if w is not None:
        return np.broadcast_to(np.asarray(w, np.float64)[p][None, :], (len(edges), C))
    return np.asarray(R, np.float64)[edges] @ np.asarray(M, np.float64)[:, p * C:(p + 1) * C]


def sh_jacobian(vec):
    """dY/dv, shape [E, 16, 3], for edge vectors vec[E, 3]."""
    vec = np.asarray(vec, dtype=np.float64).reshape(-1, 3)
    r = np.sqrt(np.einsum("ij,ij->i", vec, vec))
    ok = r * r >= 1e-30
    n = np.zeros_like(vec)
    n[ok] = vec[ok] / r[ok, None]
    x, y, z = n[:, 0], n[:, 1], n[:, 2]
    xy = x + 1j * y
    jac_n = np.zeros((len(vec), N_SH, 3))  # d/d(x, y, z) of the unit-sphere polynomial
    for l in range(_sh.L_MAX + 1):
        pl = _sh.legendre_polynomial(l)
        for m in range(0, l + 1):
            q = (-1.0) ** m * (pl.deriv(m) if m > 0 else pl)
            qz, dqz = q(z), q.deriv(1)(z)
            if m == 0:
                K = _sh.normalisation(l, 0)
                jac_n[:, _sh.sh_index(l, 0), 2] = K * dqz
                continue
            K = sqrt(2.0) * _sh.normalisation(l, m)
            pw = xy ** m
            dpw = m * xy ** (m - 1)           # d/dx of (x+iy)^m; d/dy is i times it
            kc, ks = _sh.sh_index(l, m), _sh.sh_index(l, -m)
            jac_n[:, kc, 0] = K * qz * dpw.real
            jac_n[:, kc, 1] = K * qz * (1j * dpw).real
            jac_n[:, kc, 2] = K * dqz * pw.real
            jac_n[:, ks, 0] = K * qz * dpw.imag
            jac_n[:, ks, 1] = K * qz * (1j * dpw).imag
            jac_n[:, ks, 2] = K * dqz * pw.imag
    proj = np.zeros((len(vec), 3, 3))
    proj[ok] = (np.eye(3)[None] - n[ok, :, None] * n[ok, None, :]) / r[ok, None, None]
    return np.einsum("eka,eab->ekb", jac_n, proj)


def layer_backward(vec, x, off, src, grad_out, w=None, R=None, M=None):
    """dict of gradients: x, w (shared) or R and M (radial), vec."""
    if (w is None) == (R is None or M is None):
        raise ValueError("give exactly one of w or (R, M)")
    off = np.asarray(off, dtype=np.int64)
    src = np.asarray(src, dtype=np.int64)
    x = np.asarray(x, np.float64)
    g = np.asarray(grad_out, np.float64)
    vec = np.asarray(vec, np.float64).reshape(-1, 3)
    n_recv = len(off) - 1
    C = x.shape[1]
    edges = np.arange(off[0], off[-1])
    dst = np.repeat(np.arange(n_recv), np.diff(off))
    Y = _sh.real_sh(vec[edges])
    xs, gd = x[src[edges]], g[dst]
    gx = np.zeros_like(x)
    dY = np.zeros((len(edges), N_SH))
    s = np.zeros((len(edges), len(_cg.paths()), C))
    for p, (l1, l2, l3, cr) in enumerate(_cg.real_cg_tables()):
        W = _weights(p, C, edges, w, R, M)                          # [e, C]
        b1, b2, b3 = _block(l1), _block(l2), _block(l3)
        # dL/dx: sum over k3, k2 of C g Y, weighted, scattered to senders
        t1 = np.einsum("kab,eck,eb->eca", cr, gd[:, :, b3], Y[:, b2], optimize=True)
        np.add.at(gx[:, :, b1], src[edges], W[:, :, None] * t1)
        # s: full contraction per edge, path and channel
        s[:, p, :] = np.einsum("kab,eck,eca,eb->ec", cr, gd[:, :, b3], xs[:, :, b1], Y[:, b2],
                               optimize=True)
        # dY: sum over c, k3, k1
        dY[:, b2] += np.einsum("kab,eck,eca,ec->eb", cr, gd[:, :, b3], xs[:, :, b1], W,
                               optimize=True)
    out = {"x": gx}
    if w is not None:
        out["w"] = s.sum(axis=0)
    else:
        Rm = np.asarray(R, np.float64)
        Mm = np.asarray(M, np.float64)
        sf = s.reshape(len(edges), -1)                              # column p*C + c
        gR = np.zeros_like(Rm)
        gR[edges] = sf @ Mm.T
        out["R"] = gR
        out["M"] = Rm[edges].T @ sf
    gv = np.zeros_like(vec)
    gv[edges] = np.einsum("ek,ekb->eb", dY, sh_jacobian(vec[edges]))
    out["vec"] = gv
    return out
