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
