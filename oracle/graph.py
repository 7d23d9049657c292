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

Periodic boundaries.  E2Former-V2 (section 4.2) handles periodic systems by
expanding the cells, one image per direction.  Reading: an orthorhombic box
of sides L = (L_x, L_y, L_z), positions inside it (0 <= p_a < L_a), and the
directed edges

    (sender j, image s) -> receiver i   for every s in {-1, 0, 1}^3 and every
                                        j with |p_j + s L - p_i| < r_c,
                                        except j = i with s = 0,

with d_a = (p_j[a] - p_i[a]) + s_a L_a (two float32 operations, s_a L_a
exact), d2 and the test as above, vec = d.  One image per direction is all
there is when r_c <= min(L) (a shift of 2 puts every image at least L away),
which is required.  Several images of one sender can be edges of the same
receiver (r_c > L/2); each is its own edge.  Rows are sorted by sender,
then by the image index sigma = (s_x + 1) + 3 (s_y + 1) + 9 (s_z + 1).  With
s = 0 the arithmetic is the open-boundary one, bit for bit.
  radius_graph_pbc_bruteforce  every (pair, image), chunked (small N);
  radius_graph_pbc             candidate pairs from scipy's periodic k-d
                               tree (minimum-image distance, a library
                               primitive) at a slightly larger radius, then
                               every image of each candidate pair tested.
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


# ---------------------------------------------------------------- periodic
# image shifts in index order sigma = (s_x + 1) + 3 (s_y + 1) + 9 (s_z + 1)
SHIFTS = np.array([(sx, sy, sz) for sz in (-1, 0, 1) for sy in (-1, 0, 1) for sx in (-1, 0, 1)],
                  dtype=np.int64)
SELF_IMAGE = 13  # sigma of s = (0, 0, 0)


def _box(pos, cutoff, box):
    box = np.asarray(box, dtype=_F32).reshape(3)
    if not np.all(np.isfinite(box)) or np.any(box <= 0):
        raise ValueError("box sides must be positive")
    if _F32(cutoff) > np.min(box):
        raise ValueError("the cutoff must not exceed the smallest box side")
    if len(pos) and (np.any(pos < 0) or np.any(pos >= box[None, :])):
        raise ValueError("positions must lie inside the box, 0 <= p < L")
    return box


def _image_vec(pi, pj, sL):
    """float32 d = (p_j - p_i) + s L, each operation rounded on its own."""
    return ((pj - pi).astype(_F32) + sL).astype(_F32)


def _d2v(d):
    return (d[..., 0] * d[..., 0] + d[..., 1] * d[..., 1]) + d[..., 2] * d[..., 2]


def _csr_pbc(dst, src, img, n, pos, box):
    order = np.lexsort((img, src, dst))
    dst, src, img = dst[order], src[order], img[order]
    off = np.searchsorted(dst, np.arange(n + 1), side="left").astype(np.int64)
    sL = (SHIFTS[img].astype(_F32) * box[None, :]).astype(_F32)
    vec = _image_vec(pos[dst], pos[src], sL)
    return dict(off=off, src=src.astype(np.int64), dst=dst.astype(np.int64), img=img.astype(np.int64), vec=vec)


def radius_graph_pbc_bruteforce(pos, cutoff, box, chunk=128):
    """Every (receiver, sender, image) tested; dict(off, src, dst, img, vec)."""
    pos = np.ascontiguousarray(pos, dtype=_F32).reshape(-1, 3)
    n = len(pos)
    box = _box(pos, cutoff, box)
    rc2 = _rc2(cutoff)
    dsts, srcs, imgs = [], [], []
    for k, s in enumerate(SHIFTS):
        sL = (s.astype(_F32) * box).astype(_F32)
        for a in range(0, n, chunk):
            d = _image_vec(pos[a:a + chunk, None, :], pos[None, :, :], sL)
            ii, jj = np.nonzero(_d2v(d) < rc2)
            ii = ii + a
            keep = (ii != jj) | (k != SELF_IMAGE)
            dsts.append(ii[keep])
            srcs.append(jj[keep])
            imgs.append(np.full(int(keep.sum()), k, np.int64))
    cat = lambda x: np.concatenate(x) if x else np.zeros(0, np.int64)
    return _csr_pbc(cat(dsts), cat(srcs), cat(imgs), n, pos, box)


def radius_graph_pbc(pos, cutoff, box):
    """Same set as radius_graph_pbc_bruteforce, candidate pairs from a
    periodic k-d tree: a pair with any image inside the cutoff has its
    minimum-image distance inside it too."""
    from scipy.spatial import cKDTree

    pos = np.ascontiguousarray(pos, dtype=_F32).reshape(-1, 3)
    n = len(pos)
    box = _box(pos, cutoff, box)
    rc2 = _rc2(cutoff)
    if n == 0:
        z = np.zeros(0, np.int64)
        return _csr_pbc(z, z, z, 0, pos, box)
    r_search = float(cutoff) * (1.0 + 1e-3) + 1e-3 + 1e-5 * float(np.max(box))
    tree = cKDTree(pos.astype(np.float64), boxsize=box.astype(np.float64))
    pairs = tree.query_pairs(r_search, output_type="ndarray").reshape(-1, 2).astype(np.int64)
    i = np.concatenate([pairs[:, 0], pairs[:, 1]])
    j = np.concatenate([pairs[:, 1], pairs[:, 0]])
    dsts, srcs, imgs = [], [], []
    for k, s in enumerate(SHIFTS):  # a sender is never its own image: r_c <= min(L)
        sL = (s.astype(_F32) * box).astype(_F32)
        keep = _d2v(_image_vec(pos[i], pos[j], sL)) < rc2
        dsts.append(i[keep])
        srcs.append(j[keep])
        imgs.append(np.full(int(keep.sum()), k, np.int64))
    return _csr_pbc(np.concatenate(dsts), np.concatenate(srcs), np.concatenate(imgs), n, pos, box)
