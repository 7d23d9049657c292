"""GPU parity of eqmp_fused_so2 (aligned-frame schedule) against the oracle."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import layer
from tests.gpu_util import TOL, host, oracle_kw, rel_err, to_device, weights_kw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eq():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as m

    torch.cuda.set_device(0)
    return m


def _check(eq, wl):
    import torch

    d = to_device(wl)
    got = host(eq.eqmp_fused_so2(d["vec"], d["x"], d["off"], d["src"], **weights_kw(d)))
    torch.cuda.synchronize()
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **oracle_kw(wl))
    err = rel_err(got, want)
    assert err <= TOL[wl.storage], f"rel err {err:.3e}"
    assert eq.eqmp_device_error() == 0
    return got


@pytest.mark.parametrize("C", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("storage", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_so2_channels_dtypes_modes(eq, C, storage, mode):
    _check(eq, make_workload(n_atoms=120, cutoff=5.0, channels=C, weights=mode, storage=storage, seed=400 + C))


@pytest.mark.parametrize("name", ["radial_1k_c32", "pages_1k_c32", "tiny_64"])
def test_so2_workloads(eq, name):
    _check(eq, make_workload(name))


def test_so2_axis_aligned_and_zero_length_edges(eq):
    """Edges along +z, -z, the axes, and one of zero length."""
    from equivariant_gnn_message_gb300.inputs import Workload, csr_offsets

    rng = np.random.default_rng(0)
    pos = np.array([[0, 0, 0], [0, 0, 2.0], [0, 0, -1.5], [1.0, 0, 0], [0, 1.0, 0], [0, 0, 0], [1e-4, 0, 3]])
    n = len(pos)
    pairs = sorted((i, j) for i in range(n) for j in range(n) if i != j)
    dst = np.array([p[0] for p in pairs]); src = np.array([p[1] for p in pairs])
    C = 32
    x = rng.standard_normal((n, C, 16)).astype(np.float32)
    M = (rng.standard_normal((8, 34 * C)) / np.sqrt(8)).astype(np.float32)
    R = rng.random((len(src), 8)).astype(np.float32)
    wl = Workload(name="axes", n_atoms=n, channels=C, storage="f32",
                  vec=(pos[src] - pos[dst]).astype(np.float32), src=src.astype(np.int32),
                  dst=dst.astype(np.int32), off=csr_offsets(dst, n), x=x, x_bf16_bits=None,
                  w=None, R=R, M=M)
    _check(eq, wl)


def test_so2_deterministic(eq):
    wl = make_workload("radial_1k_c32")
    d = to_device(wl)
    a = eq.eqmp_fused_so2(d["vec"], d["x"], d["off"], d["src"], **weights_kw(d)).clone()
    b = eq.eqmp_fused_so2(d["vec"], d["x"], d["off"], d["src"], **weights_kw(d))
    assert a.equal(b)


@pytest.mark.parametrize("mode,C,storage", [("shared", 32, "f32"), ("radial", 32, "f32"),
                                            ("radial", 8, "bf16"), ("radial", 128, "f32")])
def test_so2_receivers_cut_inside_clusters(eq, mode, C, storage):
    """Receivers cut between the CTAs of a cluster: a hub of degree 3000 (cut
    across every CTA of one cluster, the middle CTAs holding only part of it),
    three of degree about 200, isolated receivers and a plain ragged graph
    around them.  Compared receiver by receiver."""
    from tests.test_gpu_parity import _custom

    rng = np.random.default_rng(5)
    n = 3600
    pos = rng.uniform(0, 40, (n, 3))
    pairs = [(0, j) for j in range(1, 3001)]
    for h in (3100, 3200, 3300):
        pairs += [(h, int(j)) for j in rng.choice(n, 200, replace=False) if j != h]
    for r in range(3400, 3600):
        pairs += [(r, int(j)) for j in rng.choice(n, int(rng.integers(0, 30)), replace=False) if j != r]
    wl = _custom(pos, pairs, C=C, storage=storage, mode=mode)
    got = _check(eq, wl).astype(np.float64)
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **oracle_kw(wl))
    deg = np.diff(wl.off)
    assert np.all(got[deg == 0] == 0.0)
    num = np.linalg.norm((got - want).reshape(n, -1), axis=1)
    den = np.linalg.norm(want.reshape(n, -1), axis=1)
    has = deg > 0
    assert np.max(num[has] / den[has]) <= (1e-4 if storage == "f32" else 2e-2)
