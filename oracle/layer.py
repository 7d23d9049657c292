"""Channelwise CG tensor product + sum into receivers (oracle).

What the path computes (Batmobile blog, "Batmobile CUDA内核优化", section
"3. 操作融合": per edge, SH of the edge vector, gather of the sender's
features, tensor product, message; the message-passing sum into the
receiver is the third of the separated operations that the fusion removes):

  out[i, c, (l3, m3)] = sum over edges e with receiver i
                          sum over paths p = (l1, l2, l3)
                            W[e, p, c] * sum_{m1, m2} C^R_p[m3, m1, m2]
                                         * x[src_e, c, (l1, m1)] * Y_e[(l2, m2)]

  with W[e, p, c] = w[p, c] (shared per-path channel weights) or
  W[e, p, c] = sum_k R[e, k] M[k, p*C + c] (per-edge radial weights).

Edges are grouped by receiver in CSR form: receiver i owns the absolute
edge indices off[i] .. off[i+1]-1 of vec / src / R.  Receivers with no
edge get zeros.  Everything is float64; x is whatever values the caller
passes (for the bf16-storage workload, the bf16-rounded values).
"""
import numpy as np

from . import cg as _cg
from . import sh as _sh

N_SH = 16


def _block(l):
    return slice(l * l, (l + 1) * (l + 1))


def edge_weights(p_index, C, edges, w=None, R=None, M=None):
    """W[e, c] for path p on the given edges."""
    if w is not None:
        return np.broadcast_to(np.asarray(w, np.float64)[p_index][None, :],
                               (len(edges), C))
    Rm = np.asarray(R, np.float64)[edges]                       # [e, K]
    Mp = np.asarray(M, np.float64)[:, p_index * C:(p_index + 1) * C]  # [K, C]
    return Rm @ Mp


def _l_max(x):
    """Degree of a feature array [.., C, (l_max+1)^2]."""
    n = int(np.asarray(x).shape[-1])
    l_max = int(round(np.sqrt(n))) - 1
    if (l_max + 1) ** 2 != n:
        raise ValueError(f"{n} components is not (l_max+1)^2")
    return l_max


def edge_messages(vec, x, src, edges, w=None, R=None, M=None):
    """m[e, c, (l_max+1)^2] for the listed edge indices (definition, per path).

    The degree comes from x's last axis: 16 components is the l <= 3 layer;
    (l_max+1)^2 components the same layer over all paths with l <= l_max.
    """
    x = np.asarray(x, np.float64)
    C = x.shape[1]
    l_max = _l_max(x)
    edges = np.asarray(edges, dtype=np.int64)
    Y = _sh.real_sh(np.asarray(vec, np.float64)[edges], l_max)   # [e, (l_max+1)^2]
    xs = x[np.asarray(src)[edges]]                                # [e, C, (l_max+1)^2]
    msg = np.zeros((len(edges), C, x.shape[2]))
    for p, (l1, l2, l3, cr) in enumerate(_cg.real_cg_tables(l_max)):
        t = np.einsum("kab,eca,eb->eck", cr, xs[:, :, _block(l1)],
                      Y[:, _block(l2)], optimize=True)
        msg[:, :, _block(l3)] += edge_weights(p, C, edges, w, R, M)[:, :, None] * t
    return msg


def message_pass(vec, x, off, src, w=None, R=None, M=None, receivers=None,
                 chunk_edges=200_000):
    """out[len(receivers), C, (l_max+1)^2] (float64) for the chosen receivers
    (16 components for the l <= 3 layer).

    ``receivers`` defaults to all N = len(off) - 1.  Receivers are
    evaluated a group at a time (at most ``chunk_edges`` edges per group)
    only to bound memory; each output is the plain sum of its own edges'
    messages.
    """
    if (w is None) == (R is None or M is None):
        raise ValueError("give exactly one of w or (R, M)")
    off = np.asarray(off, dtype=np.int64)
    x = np.asarray(x, np.float64)
    C = x.shape[1]
    if receivers is None:
        receivers = np.arange(len(off) - 1)
    receivers = np.asarray(receivers, dtype=np.int64)
    out = np.zeros((len(receivers), C, x.shape[2]))
    start = 0
    while start < len(receivers):
        stop, n_e = start, 0
        while stop < len(receivers) and (stop == start or n_e < chunk_edges):
            r = receivers[stop]
            n_e += off[r + 1] - off[r]
            stop += 1
        group = receivers[start:stop]
        counts = off[group + 1] - off[group]
        edges = np.concatenate([np.arange(off[r], off[r + 1]) for r in group]) \
            if counts.sum() else np.zeros(0, np.int64)
        if len(edges):
            msg = edge_messages(vec, x, src, edges, w, R, M)
            owner = np.repeat(np.arange(len(group)), counts)
            np.add.at(out[start:stop], owner, msg)
        start = stop
    return out
