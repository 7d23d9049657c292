"""Radius graph (oracle; test infrastructure only).

What it computes.  E2Former-V2 (section 4.2, deployment notes) builds the
neighbour list by a radius cutoff rather than by a fixed k nearest
neighbours; the Batmobile blog (monitoring section) puts the cutoff at
4-6 Angstrom.  The graph is the set of directed edges

    sender j -> receiver i   for every ordered pair i != j with |p_j - p_i| < r_c,

sorted by receiver, then sender (CSR rows, receiver i owns
off[i] .. off[i+1]-1), with the edge vector vec = p_j - p_i (receiver to
sender).  Open boundaries: no periodic images.

Precision of the decision.  Whether a pair is an edge is an integer result
decided by floating point, so it is taken in the precision the GPU library
takes it, float32, in one fixed order of operations:

    d_a  = p_j[a] - p_i[a]                 a = x, y, z   (float32 subtract)
    d2   = (d_x*d_x + d_y*d_y) + d_z*d_z                 (float32 multiply, add)
    edge  iff  d2 < r_c*r_c                              (float32 product, strict)

with every operation rounded to float32 on its own (no fused multiply-add).
vec is the same float32 subtraction.  The pages fix no precision; this
reading is the plainest one that makes the edge set exact on both sides.

Two routes to the same set:
  radius_graph_bruteforce  every ordered pair, chunked over receivers
                           (small N);
  radius_graph             candidate pairs from scipy's k-d tree at a
                           slightly larger radius (a library primitive used
                           as a step), then the float32 test above.
"""
import numpy as np

_F32 = np.float32


def _rc2(cutoff):
    rc = _F32(cutoff)
    return _F32(rc * rc)


def _d2(pi, pj):
    """float32 squared distance in the fixed order, rows of pi against pj."""
    d = (pj - pi).astype(_F32)
    return (d[..., 0] * d[..., 0] + d[..., 1] * d[..., 1]) + d[..., 2] * d[..., 2]


def _csr(dst, src, n):
    order = np.lexsort((src, dst))
    dst, src = dst[order], src[order]
    off = np.searchsorted(dst, np.arange(n + 1), side="left").astype(np.int64)
    return off, src.astype(np.int64), dst.astype(np.int64)


def _finish(pos, off, src, dst):
    vec = (pos[src] - pos[dst]).astype(_F32)
    return dict(off=off, src=src, dst=dst, vec=vec)


def radius_graph_bruteforce(pos, cutoff, chunk=256):
    """Every ordered pair i != j tested; returns dict(off, src, dst, vec)."""
    pos = np.ascontiguousarray(pos, dtype=_F32).reshape(-1, 3)
    n = len(pos)
    rc2 = _rc2(cutoff)
    dsts, srcs = [], []
    for a in range(0, n, chunk):
        pi = pos[a:a + chunk, None, :]
        d2 = _d2(pi, pos[None, :, :])                     # [chunk, n]
        ii, jj = np.nonzero(d2 < rc2)
        ii = ii + a
        keep = ii != jj
        dsts.append(ii[keep])
        srcs.append(jj[keep])
    dst = np.concatenate(dsts) if dsts else np.zeros(0, np.int64)
    src = np.concatenate(srcs) if srcs else np.zeros(0, np.int64)
    off, src, dst = _csr(dst, src, n)
    return _finish(pos, off, src, dst)


def radius_graph(pos, cutoff):
    """Same set as radius_graph_bruteforce, candidates from a k-d tree."""
    from scipy.spatial import cKDTree

    pos = np.ascontiguousarray(pos, dtype=_F32).reshape(-1, 3)
    n = len(pos)
    rc2 = _rc2(cutoff)
    if n == 0:
        return _finish(pos, np.zeros(1, np.int64), np.zeros(0, np.int64), np.zeros(0, np.int64))
    # The float32 distance differs from the exact one by a few ulps of the
    # coordinates; a 1e-3 relative margin (plus 1e-3 absolute) keeps every
    # float32 edge among the candidates.
    scale = float(np.max(np.abs(pos))) if n else 0.0
    r_search = float(cutoff) * (1.0 + 1e-3) + 1e-3 + 1e-5 * scale
    pairs = cKDTree(pos.astype(np.float64)).query_pairs(r_search, output_type="ndarray")
    pairs = pairs.reshape(-1, 2).astype(np.int64)
    i = np.concatenate([pairs[:, 0], pairs[:, 1]])
    j = np.concatenate([pairs[:, 1], pairs[:, 0]])
    keep = _d2(pos[i], pos[j]) < rc2
    off, src, dst = _csr(i[keep], j[keep], n)
    return _finish(pos, off, src, dst)
