"""Pins for the radius-graph oracle (CPU only).

Fixed by things other than the oracle itself: closed-form edge counts of a
simple cubic lattice, scipy's k-d tree pair query in float64 (a library
routine; the two may differ only on pairs within rounding of the cutoff),
coincident points, and the symmetry of the relation.
"""
import numpy as np
import pytest

from oracle import graph


def _lattice(n, a=1.0):
    g = np.arange(n, dtype=np.float32) * np.float32(a)
    return np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)


def _counts(n):
    """Directed edge counts of an n^3 cubic lattice by shell (spacing 1)."""
    axis = 6 * n * n * (n - 1)                # 3 directions x n^2 (n-1) pairs x 2
    face = 12 * n * (n - 1) ** 2              # 3 planes x 2 diagonals x n (n-1)^2 x 2
    body = 8 * (n - 1) ** 3                   # 4 diagonals x (n-1)^3 x 2
    return axis, face, body


@pytest.mark.parametrize("route", [graph.radius_graph, graph.radius_graph_bruteforce])
def test_lattice_closed_form_counts(route):
    n = 6
    pos = _lattice(n)
    axis, face, body = _counts(n)
    assert len(route(pos, 1.2)["src"]) == axis
    assert len(route(pos, 1.5)["src"]) == axis + face
    assert len(route(pos, 1.8)["src"]) == axis + face + body
    # strict inequality: at exactly the spacing nothing is an edge, one ulp
    # above it the six axis neighbours are
    assert len(route(pos, 1.0)["src"]) == 0
    assert len(route(pos, np.nextafter(np.float32(1.0), np.float32(2.0)))["src"]) == axis


def test_interior_degree_is_six():
    n = 5
    g = graph.radius_graph(_lattice(n), 1.2)
    deg = np.diff(g["off"])
    idx = np.arange(n ** 3).reshape(n, n, n)
    assert np.all(deg[idx[1:-1, 1:-1, 1:-1].ravel()] == 6)
    assert np.all(deg[idx[0, 0, 0]] == 3)


def test_two_routes_agree_bitwise():
    rng = np.random.default_rng(11)
    for n, side, rc in [(700, 26.0, 5.0), (400, 8.0, 3.0), (1, 1.0, 1.0), (0, 1.0, 1.0)]:
        pos = rng.uniform(0, side, (n, 3)).astype(np.float32)
        a = graph.radius_graph(pos, rc)
        b = graph.radius_graph_bruteforce(pos, rc)
        for k in ("off", "src", "dst"):
            assert np.array_equal(a[k], b[k])
        assert np.array_equal(a["vec"].view(np.uint32), b["vec"].view(np.uint32))


def test_matches_scipy_pairs_up_to_rounding_at_the_cutoff():
    from scipy.spatial import cKDTree

    rng = np.random.default_rng(5)
    pos = rng.uniform(0, 30.0, (1500, 3)).astype(np.float32)
    rc = 5.0
    g = graph.radius_graph(pos, rc)
    ours = set(zip(g["dst"].tolist(), g["src"].tolist()))
    pairs = cKDTree(pos.astype(np.float64)).query_pairs(rc, output_type="ndarray")
    ref = set(map(tuple, pairs.tolist())) | set(map(tuple, pairs[:, ::-1].tolist()))
    diff = ours ^ ref
    assert len(ours) > 10_000
    for i, j in diff:
        d = np.linalg.norm(pos[i].astype(np.float64) - pos[j].astype(np.float64))
        assert abs(d - rc) < 1e-5 * rc


def test_relation_is_symmetric_sorted_and_loop_free():
    rng = np.random.default_rng(3)
    pos = rng.uniform(0, 20.0, (600, 3)).astype(np.float32)
    g = graph.radius_graph(pos, 4.0)
    src, dst = g["src"], g["dst"]
    assert np.all(src != dst)
    assert set(zip(src.tolist(), dst.tolist())) == set(zip(dst.tolist(), src.tolist()))
    assert np.all(np.diff(dst) >= 0)
    same = np.diff(dst) == 0
    assert np.all(np.diff(src)[same] > 0)
    assert np.array_equal(g["vec"], (pos[src] - pos[dst]).astype(np.float32))
    assert np.array_equal(np.repeat(np.arange(600), np.diff(g["off"])), dst)


def test_coincident_points_form_a_complete_graph():
    pos = np.full((40, 3), 1.25, np.float32)
    g = graph.radius_graph(pos, 0.5)
    assert len(g["src"]) == 40 * 39
    assert np.all(g["vec"] == 0)


def test_planted_non_strict_cutoff_fails_the_lattice_count():
    """A '<=' slipped into the test would count the axis shell at r_c = a."""
    pos = _lattice(4)
    d2 = graph._d2(pos[:, None, :], pos[None, :, :])
    loose = int(np.sum(d2 <= graph._rc2(1.0))) - len(pos)
    assert loose == _counts(4)[0]
    assert len(graph.radius_graph_bruteforce(pos, 1.0)["src"]) == 0


# ---------------------------------------------------------------- periodic
_PBC_ROUTES = [graph.radius_graph_pbc, graph.radius_graph_pbc_bruteforce]


@pytest.mark.parametrize("route", _PBC_ROUTES)
@pytest.mark.parametrize("n", [2, 3, 5])
def test_pbc_lattice_every_site_has_the_bulk_shells(route, n):
    """A periodic n^3 lattice has no surface: every site sees 6, 18, 26
    neighbours (axis, + face diagonals, + body diagonals).  At n = 2 these
    come from fewer atoms, several images each."""
    pos = _lattice(n)
    box = (n, n, n)
    for rc, per_site in ((1.2, 6), (1.5, 18), (1.8, 26)):
        g = route(pos, rc, box)
        assert np.all(np.diff(g["off"]) == per_site)
        # every edge vector is a lattice vector of the shell's length
        d2 = np.sum(g["vec"].astype(np.float64) ** 2, axis=1)
        assert np.all(d2 < rc * rc) and np.all(d2 >= 1.0)
    assert len(route(pos, 1.0, box)["src"]) == 0  # strict at the spacing
    assert len(route(pos, np.nextafter(np.float32(1.0), np.float32(2.0)), box)["src"]) == 6 * n ** 3


def test_pbc_two_routes_agree_bitwise():
    rng = np.random.default_rng(12)
    # bulk density; a box just above the cutoff (several images of a sender);
    # anisotropic; one atom; none
    for n, box, rc in [(700, (26.0, 26.0, 26.0), 5.0), (60, (5.5, 7.0, 6.0), 5.0),
                       (300, (30.0, 8.0, 12.0), 4.0), (1, (3.0, 3.0, 3.0), 2.0), (0, (3.0, 3.0, 3.0), 2.0)]:
        pos = (rng.uniform(0, 1, (n, 3)) * np.asarray(box)).astype(np.float32)
        pos = np.minimum(pos, np.nextafter(np.asarray(box, np.float32), np.float32(0)))
        a = graph.radius_graph_pbc(pos, rc, box)
        b = graph.radius_graph_pbc_bruteforce(pos, rc, box)
        for k in ("off", "src", "dst", "img"):
            assert np.array_equal(a[k], b[k]), k
        assert np.array_equal(a["vec"].view(np.uint32), b["vec"].view(np.uint32))


def test_pbc_in_a_box_far_larger_than_the_cluster_is_the_open_graph():
    """No image is in reach: the periodic graph is the open one, bit for bit."""
    rng = np.random.default_rng(13)
    pos = rng.uniform(100.0, 120.0, (500, 3)).astype(np.float32)
    a = graph.radius_graph_pbc(pos, 4.0, (400.0, 400.0, 400.0))
    b = graph.radius_graph(pos, 4.0)
    assert np.all(a["img"] == graph.SELF_IMAGE)
    for k in ("off", "src", "dst"):
        assert np.array_equal(a[k], b[k])
    assert np.array_equal(a["vec"].view(np.uint32), b["vec"].view(np.uint32))


def test_pbc_every_edge_has_its_exact_reverse():
    """(i <- j, s) and (j <- i, -s) are both edges with opposite vectors, bit
    for bit (negation is exact and the rounding is symmetric)."""
    rng = np.random.default_rng(14)
    box = (9.0, 7.0, 11.0)
    pos = (rng.uniform(0, 1, (200, 3)) * np.asarray(box)).astype(np.float32)
    g = graph.radius_graph_pbc(pos, 5.0, box)
    trip = list(zip(g["dst"].tolist(), g["src"].tolist(), g["img"].tolist()))
    idx = {t: e for e, t in enumerate(trip)}
    assert len(idx) == len(trip)  # (receiver, sender, image) unique
    rev = np.array([idx[(s, d, 26 - m)] for d, s, m in trip])
    assert np.array_equal(g["vec"][rev].view(np.uint32), (-g["vec"]).view(np.uint32))
    assert np.array_equal(rev[rev], np.arange(len(trip)))


def test_pbc_matches_scipy_periodic_pairs_up_to_rounding():
    """With r_c <= L/2 a pair has at most one image in reach: the edge pairs
    are scipy's periodic (minimum-image) k-d tree pairs, up to pairs within
    rounding of the cutoff."""
    from scipy.spatial import cKDTree

    rng = np.random.default_rng(15)
    L = 24.0
    pos = rng.uniform(0, L, (1200, 3)).astype(np.float32)
    rc = 5.0
    g = graph.radius_graph_pbc(pos, rc, (L, L, L))
    ours = set(zip(g["dst"].tolist(), g["src"].tolist()))
    assert len(ours) == len(g["src"])  # one image per pair
    pairs = cKDTree(pos.astype(np.float64), boxsize=L).query_pairs(rc, output_type="ndarray")
    ref = set(map(tuple, pairs.tolist())) | set(map(tuple, pairs[:, ::-1].tolist()))
    assert len(ours) > 10_000
    for i, j in ours ^ ref:
        d = pos[j].astype(np.float64) - pos[i].astype(np.float64)
        d -= L * np.round(d / L)
        assert abs(np.linalg.norm(d) - rc) < 1e-5 * rc


def test_pbc_preconditions():
    pos = np.zeros((4, 3), np.float32)
    with pytest.raises(ValueError):
        graph.radius_graph_pbc(pos, 5.0, (4.0, 6.0, 6.0))       # cutoff above a side
    with pytest.raises(ValueError):
        graph.radius_graph_pbc(pos + 6.0, 3.0, (6.0, 6.0, 6.0))  # outside the box
    with pytest.raises(ValueError):
        graph.radius_graph_pbc(pos, 1.0, (0.0, 6.0, 6.0))


def test_planted_one_sided_images_fail_the_periodic_lattice():
    """Images taken in one direction only (s in {0, 1}) would give the
    surface sites of the open lattice fewer than six neighbours."""
    pos = _lattice(3)
    box = np.float32(3.0)
    rc2 = graph._rc2(1.2)
    deg = np.zeros(len(pos), int)
    for s in graph.SHIFTS:
        if np.any(s < 0):
            continue
        d = graph._image_vec(pos[:, None, :], pos[None, :, :], (s.astype(np.float32) * box).astype(np.float32))
        hit = graph._d2v(d) < rc2
        if not np.any(s):
            np.fill_diagonal(hit, False)
        deg += hit.sum(1)
    assert np.any(deg != 6)
    assert np.all(np.diff(graph.radius_graph_pbc_bruteforce(pos, 1.2, (3, 3, 3))["off"]) == 6)
