"""GPU parity of eqmp_fused_lmax (degrees 4..6, aligned-frame schedule)
against the oracle's dense layer at the same degree."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import layer
from tests.gpu_util import host, oracle_kw, rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def eq():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as m

    torch.cuda.set_device(0)
    return m


def _dev(wl):
    import torch

    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dict(vec=t(wl.vec), x=t(wl.x), off=t(wl.off), src=t(wl.src), w=t(wl.w), R=t(wl.R), M=t(wl.M))


def _run(eq, l_max, d, **over):
    kw = dict(w=d["w"]) if d["w"] is not None else dict(R=d["R"], M=d["M"])
    kw.update(over)
    return host(eq.eqmp_fused_lmax(l_max, d["vec"], d["x"], d["off"], d["src"], **kw))


def _check(eq, wl, l_max):
    import torch

    got = _run(eq, l_max, _dev(wl))
    torch.cuda.synchronize()
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **oracle_kw(wl))
    err = rel_err(got, want)
    assert err <= TOL, f"l_max {l_max}: rel err {err:.3e}"
    return got


@pytest.mark.parametrize("l_max", [4, 5, 6])
@pytest.mark.parametrize("mode", ["shared", "radial"])
@pytest.mark.parametrize("C", [8, 32, 64, 128])
def test_parity_grid(eq, l_max, mode, C):
    n = 40 if C == 128 else 60
    wl = make_workload(n_atoms=n, cutoff=5.0, channels=C, weights=mode, storage="f32", seed=30 + l_max,
                       l_max=l_max)
    _check(eq, wl, l_max)


@pytest.mark.parametrize("l_max", [4, 6])
def test_pages_sized_graph(eq, l_max):
    wl = make_workload(n_atoms=300, cutoff=5.0, channels=16, weights="shared", storage="f32", seed=41,
                       l_max=l_max)
    _check(eq, wl, l_max)


def test_path_counts(eq):
    assert [eq.eqmp_num_paths_lmax(l) for l in (3, 4, 5, 6)] == [34, 65, 111, 175]


def test_edge_cases(eq):
    """Axis-aligned and zero-length edges, empty receivers, an out-of-range sender."""
    import torch

    l_max = 5
    wl = make_workload(n_atoms=50, cutoff=5.0, channels=8, weights="radial", storage="f32", seed=44,
                       l_max=l_max)
    vec = wl.vec.copy()
    vec[0] = (0.0, 0.0, 2.0)       # along +z
    vec[1] = (0.0, 0.0, -3.0)      # along -z (the frame's other branch)
    vec[2] = (0.0, 0.0, 0.0)       # zero length
    vec[3] = (1.5, 0.0, 0.0)
    wl.vec = vec
    _check(eq, wl, l_max)
    # receivers with no edge: a CSR that skips some rows
    off = wl.off.copy()
    off[5:9] = off[5]
    d = _dev(wl)
    d["off"] = torch.from_numpy(off).cuda()
    got = _run(eq, l_max, d)
    want = layer.message_pass(wl.vec, wl.x, off, wl.src, **oracle_kw(wl))
    assert rel_err(got, want) <= TOL
    assert np.all(got[5:8] == 0.0)
    # an out-of-range sender adds nothing
    src = wl.src.copy()
    src[10] = 10_000
    d = _dev(wl)
    d["src"] = torch.from_numpy(src).cuda()
    got = _run(eq, l_max, d)
    keep = np.ones(len(src), bool)
    keep[10] = False
    R = wl.R.copy()
    R[10] = 0.0  # the oracle's view: that edge contributes zero
    want = layer.message_pass(wl.vec, wl.x, wl.off, np.where(keep, src, 0), R=R, M=wl.M)
    assert rel_err(got, want) <= TOL


def test_deterministic_and_argument_errors(eq):
    import torch

    wl = make_workload(n_atoms=80, cutoff=5.0, channels=32, weights="shared", storage="f32", seed=45, l_max=4)
    d = _dev(wl)
    a = eq.eqmp_fused_lmax(4, d["vec"], d["x"], d["off"], d["src"], w=d["w"])
    b = eq.eqmp_fused_lmax(4, d["vec"], d["x"], d["off"], d["src"], w=d["w"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    lib = eq.load_library()
    st = torch.cuda.current_stream().cuda_stream
    W = eq.Weights(d["w"].data_ptr(), None, None, 0)
    for l_max in (3, 7):
        s = lib.eqmp_fused_lmax(l_max, d["vec"].data_ptr(), d["x"].data_ptr(), 80, d["off"].data_ptr(),
                                d["src"].data_ptr(), 80, wl.n_edges, 32, W, a.data_ptr(), st)
        assert s == eq.EQMP_ERR_UNSUPPORTED
    s = lib.eqmp_fused_lmax(4, d["vec"].data_ptr(), d["x"].data_ptr(), 80, d["off"].data_ptr(),
                            d["src"].data_ptr(), 80, wl.n_edges, 24, W, a.data_ptr(), st)
    assert s == eq.EQMP_ERR_UNSUPPORTED


@pytest.mark.parametrize("l_max,C,mode", [(4, 8, "shared"), (4, 32, "radial"), (6, 32, "shared")])
def test_hub_wraps_the_rings(eq, l_max, C, mode):
    """A receiver of degree 600 (one CTA's producer batches and row ring wrap
    many times inside it) beside isolated receivers and a ragged graph,
    compared receiver by receiver."""
    from equivariant_gnn_message_gb300.inputs import Workload, csr_offsets

    rng = np.random.default_rng(46)
    n = 700
    pos = rng.uniform(0, 30, (n, 3))
    pairs = [(0, j) for j in range(1, 601)]
    for r in range(600, 700):
        pairs += [(r, int(j)) for j in rng.choice(n, int(rng.integers(0, 25)), replace=False) if j != r]
    pairs = np.asarray(sorted(pairs), dtype=np.int64)
    dst, src = pairs[:, 0], pairs[:, 1]
    nc = (l_max + 1) ** 2
    P = eq.eqmp_num_paths_lmax(l_max)
    x = rng.standard_normal((n, C, nc)).astype(np.float32)
    w = (rng.standard_normal((P, C)) / np.sqrt(P)).astype(np.float32) if mode == "shared" else None
    M = (rng.standard_normal((8, P * C)) / np.sqrt(8)).astype(np.float32) if mode != "shared" else None
    R = rng.random((len(src), 8)).astype(np.float32) if mode != "shared" else None
    wl = Workload(name="hub", n_atoms=n, channels=C, storage="f32", vec=(pos[src] - pos[dst]).astype(np.float32),
                  src=src.astype(np.int32), dst=dst.astype(np.int32), off=csr_offsets(dst, n), x=x,
                  x_bf16_bits=None, w=w, R=R, M=M)
    got = _run(eq, l_max, _dev(wl)).astype(np.float64)
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **oracle_kw(wl))
    deg = np.diff(wl.off)
    assert np.all(got[deg == 0] == 0.0)
    num = np.linalg.norm((got - want).reshape(n, -1), axis=1)
    den = np.linalg.norm(want.reshape(n, -1), axis=1)
    assert np.max(num[deg > 0] / den[deg > 0]) <= TOL
    assert eq.eqmp_device_error() == 0


def test_misaligned_features_are_rejected(eq):
    """Sender rows are bulk-copied, so x must start on a 16-byte boundary."""
    import torch

    wl = make_workload(n_atoms=40, cutoff=5.0, channels=8, weights="shared", storage="f32", seed=47, l_max=4)
    d = _dev(wl)
    lib = eq.load_library()
    buf = torch.zeros(d["x"].numel() + 4, dtype=torch.float32, device="cuda")
    out = torch.empty((40, 8, 25), dtype=torch.float32, device="cuda")
    W = eq.Weights(d["w"].data_ptr(), None, None, 0)
    st = torch.cuda.current_stream().cuda_stream
    s = lib.eqmp_fused_lmax(4, d["vec"].data_ptr(), buf.data_ptr() + 4, 40, d["off"].data_ptr(),
                            d["src"].data_ptr(), 40, wl.n_edges, 8, W, out.data_ptr(), st)
    assert s == eq.EQMP_ERR_INVALID_ARG
