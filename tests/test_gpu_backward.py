"""GPU parity of eqmp_fused_backward against the oracle's gradients."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import backward
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


def _run(eq, wl, g, need):
    import torch

    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    so, se = eq.sender_view(wl.src, wl.n_atoms)
    out = eq.eqmp_fused_backward(t(wl.vec), t(wl.x), t(wl.off), t(wl.src), t(wl.dst), t(so), t(se),
                                 t(g), w=t(wl.w), R=t(wl.R), M=t(wl.M), need=need)
    torch.cuda.synchronize()
    assert eq.eqmp_device_error() == 0
    return {k: host(v) for k, v in out.items()}


@pytest.mark.parametrize("C", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_backward_parity(eq, C, mode):
    wl = make_workload(n_atoms=60, cutoff=5.0, channels=C, weights=mode, storage="f32", seed=200 + C)
    g = np.random.default_rng(C).standard_normal((wl.n_atoms, C, 16)).astype(np.float32)
    need = ("x", "vec", "w") if mode == "shared" else ("x", "vec", "R", "M")
    got = _run(eq, wl, g, need)
    want = backward.layer_backward(wl.vec, wl.x, wl.off, wl.src, g, **oracle_kw(wl))
    for k in need:
        err = rel_err(got[k], want[k])
        assert err <= TOL, f"grad {k}: rel err {err:.3e}"


@pytest.mark.parametrize("name", ["pages_1k_c32", "radial_1k_c32"])
def test_backward_workloads(eq, name):
    wl = make_workload(name)
    g = np.random.default_rng(1).standard_normal((wl.n_atoms, wl.channels, 16)).astype(np.float32)
    need = ("x", "vec", "w") if wl.w is not None else ("x", "vec", "R", "M")
    got = _run(eq, wl, g, need)
    want = backward.layer_backward(wl.vec, wl.x, wl.off, wl.src, g, **oracle_kw(wl))
    for k in need:
        assert rel_err(got[k], want[k]) <= TOL, k


@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_backward_10k_atoms_every_gradient(eq, mode):
    """A 10,000-atom graph (about 190k edges, C = 32) in full: every row of
    dx, dvec (and dR) and every entry of dw (dM) against the oracle, which
    runs on all host cores (per receiver range, partial gradients summed)."""
    from tests import oracle_pool

    wl = make_workload(n_atoms=10_000, cutoff=5.0, channels=32, weights=mode, storage="f32", seed=210)
    g = np.random.default_rng(3).standard_normal((wl.n_atoms, 32, 16)).astype(np.float32)
    need = ("x", "vec", "w") if mode == "shared" else ("x", "vec", "R", "M")
    got = _run(eq, wl, g, need)
    want = oracle_pool.layer_backward_all(wl, g)
    for k in need:
        err = rel_err(got[k], want[k])
        print(f"backward 10k {mode} grad {k}: E={wl.n_edges} rel err {err:.3e}")
        assert err <= TOL, f"grad {k}: rel err {err:.3e}"


def test_backward_deterministic_and_skips(eq):
    wl = make_workload(n_atoms=200, cutoff=5.0, channels=32, weights="shared", storage="f32", seed=5)
    g = np.random.default_rng(2).standard_normal((wl.n_atoms, 32, 16)).astype(np.float32)
    a = _run(eq, wl, g, ("x", "vec", "w"))
    b = _run(eq, wl, g, ("x", "vec", "w"))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    only_x = _run(eq, wl, g, ("x",))
    assert np.array_equal(only_x["x"], a["x"])
