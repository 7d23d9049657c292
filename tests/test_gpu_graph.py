"""GPU parity of eqmp_radius_graph against the oracle (bit-exact: integers,
and the float32 edge vectors compared bit for bit)."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import DENSITY, make_workload
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


def _gpu(eq, pos, cutoff, **kw):
    import torch

    out, E = eq.eqmp_radius_graph(torch.from_numpy(np.ascontiguousarray(pos, np.float32)).cuda(), cutoff, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, E


def _reverse_index(off, src, dst):
    """Position of edge (src -> dst) reversed, from the oracle's CSR."""
    key = dst.astype(np.int64) * (len(off) - 1) + src          # sorted: rows by dst, src ascending
    rkey = src.astype(np.int64) * (len(off) - 1) + dst
    pos = np.searchsorted(key, rkey)
    assert np.array_equal(key[pos], rkey)
    return pos


def _same(eq, pos, cutoff, want=None):
    got, E = _gpu(eq, pos, cutoff, dst=True, rev=True)
    want = want or graph.radius_graph(pos, cutoff)
    assert E == len(want["src"])
    assert np.array_equal(got["off"], want["off"])
    assert np.array_equal(got["src"], want["src"])
    assert np.array_equal(got["dst"], want["dst"])
    assert np.array_equal(got["vec"].view(np.uint32), want["vec"].view(np.uint32))
    assert np.array_equal(got["rev"], _reverse_index(want["off"], want["src"], want["dst"]))
    return got


@pytest.mark.parametrize("name", ["tiny_64", "pages_1k_c32", "dense_10k_c128_bf16", "scale_100k_c64"])
def test_workload_graphs_bit_exact(eq, name):
    wl = make_workload(name)
    _same(eq, wl.pos, wl.cutoff)


def test_rows_past_the_scratch_length(eq):
    """The first walk keeps rows of up to 96 senders and the second walks
    again for longer ones: a dense 20,000-atom box at cutoff 9 (about 100
    neighbours, so rows on both sides of the length) and a box with a crowded
    corner (rows of a few hundred)."""
    rng = np.random.default_rng(23)
    n = 20_000
    side = (n / DENSITY) ** (1 / 3)
    pos = rng.uniform(0, side, (n, 3)).astype(np.float32)
    got = _same(eq, pos, 9.0)
    deg = np.diff(got["off"])
    assert (deg <= 96).any() and (deg > 96).any()
    pos2 = pos.copy()
    pos2[:600] = rng.uniform(0, 4.0, (600, 3)).astype(np.float32)
    got2 = _same(eq, pos2, 5.0)
    assert np.diff(got2["off"]).max() > 500


def test_single_launch_rows_past_the_scratch_length(eq):
    """The same in the single cooperative launch (3000 atoms): a crowded
    corner gives rows of a few hundred next to ordinary ones."""
    rng = np.random.default_rng(24)
    n = 3000
    side = (n / DENSITY) ** (1 / 3)
    pos = rng.uniform(0, side, (n, 3)).astype(np.float32)
    pos[:400] = rng.uniform(0, 4.0, (400, 3)).astype(np.float32)
    got = _same(eq, pos, 5.0)
    deg = np.diff(got["off"])
    assert deg.max() > 96 and (deg <= 96).any()


def test_ragged_sizes_and_negative_coordinates(eq):
    rng = np.random.default_rng(21)
    for n in (1, 2, 31, 257, 4099):
        side = (n / DENSITY) ** (1 / 3)
        pos = rng.uniform(-side, 0.3 * side, (n, 3)).astype(np.float32) - 1000.0
        _same(eq, pos, 5.0)


def test_empty_and_single_atom(eq):
    got, E = _gpu(eq, np.zeros((0, 3), np.float32), 5.0)
    assert E == 0 and np.array_equal(got["off"], [0])
    got, E = _gpu(eq, np.ones((1, 3), np.float32), 5.0)
    assert E == 0 and np.array_equal(got["off"], [0, 0])


def test_lattice_cutoff_is_strict(eq):
    g = np.arange(6, dtype=np.float32)
    pos = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    got, E = _gpu(eq, pos, 1.0)
    assert E == 0
    _same(eq, pos, float(np.nextafter(np.float32(1.0), np.float32(2.0))))
    _same(eq, pos, 1.5)


def test_coincident_points_and_long_rows(eq):
    """700 atoms at one point: rows of 699 edges take the long-row sort."""
    pos = np.full((700, 3), 3.5, np.float32)
    got = _same(eq, pos, 0.5)
    assert len(got["src"]) == 700 * 699


def test_cluster_with_hub(eq):
    rng = np.random.default_rng(4)
    far = rng.uniform(0, 60.0, (3000, 3))
    ball = rng.normal(30.0, 0.4, (900, 3))                     # a dense clump: rows of hundreds
    pos = np.concatenate([far, ball]).astype(np.float32)
    _same(eq, pos, 2.0, want=graph.radius_graph_bruteforce(pos, 2.0))


def test_capacity_too_small_reports_the_count(eq):
    import torch

    wl = make_workload("tiny_64")
    lib = eq.load_library()
    pos = torch.from_numpy(wl.pos).cuda()
    N = len(wl.pos)
    ws = torch.empty(lib.eqmp_radius_graph_workspace_size(N), dtype=torch.uint8, device="cuda")
    off = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    e = torch.empty(1, dtype=torch.int64, device="cuda")
    src = torch.empty(10, dtype=torch.int32, device="cuda")
    vec = torch.empty((10, 3), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for cap in (10, 0):
        s = lib.eqmp_radius_graph(pos.data_ptr(), N, wl.cutoff, off.data_ptr(), src.data_ptr(), vec.data_ptr(),
                                  None, None, cap, e.data_ptr(), ws.data_ptr(), ws.numel(), st)
        assert s == eq.EQMP_OK
        torch.cuda.synchronize()
        want = graph.radius_graph(wl.pos, wl.cutoff)
        assert int(e.item()) == len(want["src"])
        assert np.array_equal(off.cpu().numpy(), want["off"])
    # the binding's retry path with a small first capacity
    got, E = _gpu(eq, wl.pos, wl.cutoff, e_cap=5)
    assert np.array_equal(got["src"], want["src"])


def test_bad_positions_and_arguments(eq):
    pos = np.zeros((50, 3), np.float32)
    pos[:, 0] = np.arange(50)
    bad = pos.copy()
    bad[7, 1] = np.nan
    with pytest.raises(eq.EqmpError):
        _gpu(eq, bad, 2.0)
    far = pos.copy()
    far[3, 2] = 1e9
    with pytest.raises(eq.EqmpError):
        _gpu(eq, far, 2.0)
    for cutoff in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(eq.EqmpError):
            _gpu(eq, pos, cutoff)
    # the context is still usable
    _same(eq, pos, 2.0)


def test_deterministic(eq):
    wl = make_workload("pages_1k_c32")
    a, _ = _gpu(eq, wl.pos, wl.cutoff, dst=True, rev=True)
    b, _ = _gpu(eq, wl.pos, wl.cutoff, dst=True, rev=True)
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8))


def test_graph_feeds_the_layer_and_its_backward(eq):
    """GPU graph -> eqmp_fused matches the oracle layer on the oracle graph;
    (row_offsets, rev) is the sender view the backward takes."""
    import torch

    wl = make_workload("pages_1k_c32")
    out, E = eq.eqmp_radius_graph(torch.from_numpy(wl.pos).cuda(), wl.cutoff, dst=True, rev=True)
    x = torch.from_numpy(wl.x).cuda()
    w = torch.from_numpy(wl.w).cuda()
    got = host(eq.eqmp_fused(out["vec"], x, out["off"], out["src"], w=w))
    g = graph.radius_graph(wl.pos, wl.cutoff)
    want = layer.message_pass(g["vec"], wl.x, g["off"], g["src"], w=wl.w)
    assert rel_err(got, want) <= 1e-4
    so, se = eq.sender_view(g["src"], len(wl.pos))
    assert np.array_equal(out["off"].cpu().numpy(), so)
    assert np.array_equal(out["rev"].cpu().numpy(), se)
    gout = torch.randn(out["off"].shape[0] - 1, wl.channels, 16, device="cuda")
    a = eq.eqmp_fused_backward(out["vec"], x, out["off"], out["src"], out["dst"], out["off"], out["rev"], gout, w=w)
    b = eq.eqmp_fused_backward(out["vec"], x, out["off"], out["src"], out["dst"], torch.from_numpy(so).cuda(),
                               torch.from_numpy(se).cuda(), gout, w=w)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert eq.eqmp_device_error() == 0
