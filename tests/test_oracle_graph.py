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
