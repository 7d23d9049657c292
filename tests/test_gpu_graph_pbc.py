"""GPU parity of eqmp_radius_graph_pbc (periodic boundaries) against the
oracle: offsets, senders, image indices, receivers and reverse edges bit
for bit, the float32 edge vectors compared bit for bit."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import DENSITY
from oracle import graph, layer
from tests.gpu_util import host, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eq():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as m

    torch.cuda.set_device(0)
    return m


def _inside(pos, box):
    """Positions strictly inside [0, L) (float32)."""
    top = np.nextafter(np.asarray(box, np.float32), np.float32(0))
    return np.minimum(np.maximum(pos.astype(np.float32), np.float32(0)), top)


def _gpu(eq, pos, cutoff, box, **kw):
    import torch

    out, E = eq.eqmp_radius_graph(torch.from_numpy(np.ascontiguousarray(pos, np.float32)).cuda(), cutoff,
                                  box=box, **kw)
    torch.cuda.synchronize()
    assert eq.eqmp_device_error() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}, E


def _reverse_index(want):
    n = len(want["off"]) - 1
    key = (want["dst"] * n + want["src"]) * 27 + want["img"]          # sorted by construction
    rkey = (want["src"] * n + want["dst"]) * 27 + (26 - want["img"])
    at = np.searchsorted(key, rkey)
    assert np.array_equal(key[at], rkey)
    return at


def _same(eq, pos, cutoff, box):
    got, E = _gpu(eq, pos, cutoff, box, dst=True, rev=True)
    want = graph.radius_graph_pbc(pos, cutoff, box)
    assert E == len(want["src"])
    for k in ("off", "src", "img", "dst"):
        assert np.array_equal(got[k], want[k]), k
    assert np.array_equal(got["vec"].view(np.uint32), want["vec"].view(np.uint32))
    assert np.array_equal(got["rev"], _reverse_index(want))
    return got, want


@pytest.mark.parametrize("n", [64, 1000, 10_000, 30_000])
def test_bulk_density_bit_exact(eq, n):
    """The workloads' density in a periodic cube: up to 16,384 atoms the
    single cooperative launch, above it the multi-kernel path."""
    L = (n / DENSITY) ** (1 / 3)
    pos = _inside(np.random.default_rng(n).uniform(0, L, (n, 3)), (L, L, L))
    got, want = _same(eq, pos, 5.0, (L, L, L))
    if n >= 1000:  # no surface: about the bulk neighbour count
        assert abs(len(want["src"]) / n - DENSITY * 4 / 3 * np.pi * 125) < 1.0


@pytest.mark.parametrize("box", [(5.5, 7.0, 6.0), (5.0, 5.0, 5.0), (30.0, 8.0, 12.0), (16.0, 5.2, 40.0)])
def test_small_and_anisotropic_boxes(eq, box):
    """Sides below three cells (one cell, its images walked explicitly),
    the cutoff equal to a side, and a sender in reach through several of
    its images."""
    n = max(8, int(DENSITY * np.prod(box)))
    pos = _inside(np.random.default_rng(int(sum(box))).uniform(0, 1, (n, 3)) * np.asarray(box), box)
    got, want = _same(eq, pos, 5.0, box)
    if box[0] < 10.0:
        rows = np.repeat(np.arange(n), np.diff(want["off"]))
        _, counts = np.unique(rows * n + want["src"], return_counts=True)
        assert counts.max() > 1  # some sender appears under several images


@pytest.mark.parametrize("m", [2, 3, 5])
def test_lattice_shells(eq, m):
    g = np.arange(m, dtype=np.float32)
    pos = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    for rc, per in ((1.2, 6), (1.5, 18), (1.8, 26)):
        got, _ = _same(eq, pos, rc, (m, m, m))
        assert np.all(np.diff(got["off"]) == per)
    got, E = _gpu(eq, pos, 1.0, (m, m, m))
    assert E == 0


def test_large_box_is_the_open_graph(eq):
    pos = np.random.default_rng(31).uniform(100.0, 120.0, (800, 3)).astype(np.float32)
    got, _ = _gpu(eq, pos, 4.0, (400.0, 400.0, 400.0))
    opn, _ = _gpu(eq, pos, 4.0, None)
    assert np.all(got["img"] == 13)
    for k in ("off", "src"):
        assert np.array_equal(got[k], opn[k])
    assert np.array_equal(got["vec"].view(np.uint32), opn["vec"].view(np.uint32))


def test_empty_single_and_errors(eq):
    import torch

    got, E = _gpu(eq, np.zeros((0, 3), np.float32), 5.0, (10.0, 10.0, 10.0))
    assert E == 0 and np.array_equal(got["off"], [0])
    got, E = _gpu(eq, np.ones((1, 3), np.float32), 5.0, (10.0, 10.0, 10.0))
    assert E == 0 and np.array_equal(got["off"], [0, 0])
    p = torch.ones((4, 3), device="cuda")
    with pytest.raises(eq.EqmpError) as ei:  # cutoff above a side
        eq.eqmp_radius_graph(p, 5.0, box=(4.0, 10.0, 10.0))
    assert ei.value.status == eq.EQMP_ERR_UNSUPPORTED
    with pytest.raises(eq.EqmpError) as ei:  # a non-positive side
        eq.eqmp_radius_graph(p, 1.0, box=(0.0, 10.0, 10.0))
    assert ei.value.status == eq.EQMP_ERR_INVALID_ARG
    with pytest.raises(eq.EqmpError) as ei:  # an atom outside the box: E = -1, no fault
        eq.eqmp_radius_graph(p * 12.0, 1.0, box=(10.0, 10.0, 10.0))
    assert ei.value.status == eq.EQMP_ERR_INVALID_ARG
    assert eq.eqmp_device_error() == 0


def test_layer_on_a_periodic_graph_matches_the_oracle(eq):
    """The fused layer takes a periodic graph as it comes (a sender may
    appear under several images, each edge with its own vector)."""
    import torch

    rng = np.random.default_rng(41)
    box = (9.0, 8.0, 10.0)
    n = 40
    pos = _inside(rng.uniform(0, 1, (n, 3)) * np.asarray(box), box)
    g = graph.radius_graph_pbc(pos, 5.0, box)
    C = 32
    x = rng.standard_normal((n, C, 16)).astype(np.float32)
    w = (rng.standard_normal((34, C)) / np.sqrt(34)).astype(np.float32)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).astype(dt)).cuda()
    got = host(eq.eqmp_fused(t(g["vec"], np.float32), t(x, np.float32), t(g["off"], np.int32),
                             t(g["src"], np.int32), w=t(w, np.float32)))
    want = layer.message_pass(g["vec"], x, g["off"], g["src"], w=w)
    assert rel_err(got, want) <= 1e-4


@pytest.mark.parametrize("n", [3000, 20_000])
def test_crowded_rows_past_the_scratch_length(eq, n):
    """Rows longer than the 96-sender scratch of the first walk, in the
    single launch (3000 atoms) and in the separate launches (20,000): a
    crowded region straddling a box face, so its long rows hold senders
    under several images."""
    rng = np.random.default_rng(31 + n)
    side = float((n / DENSITY) ** (1 / 3))
    box = (side, side, side)
    pos = rng.uniform(0, side, (n, 3))
    crowd = rng.uniform(-2.0, 2.0, (400, 3)) + np.array([0.0, side / 2, side / 2])
    pos[:400] = np.mod(crowd, side)
    pos = _inside(pos, box)
    got, _ = _same(eq, pos, 5.0, box)
    assert np.diff(got["off"]).max() > 96
