"""The aligned-frame (SO(2)) schedule of the build-time generator
reproduces the oracle's dense layer (CPU only).

E2Former-V2 (section 2.1, Lemma 4.1 and Eq. 13): rotate the sender features
into a frame whose z axis is the edge, where the edge harmonics keep only
m = 0 and each output order takes one input order; rotate back.  This checks
the generator's frame, Wigner-D recursion and aligned-frame term table, which
the CUDA kernel of eqmp_fused_so2 uses, against the plain definition.
"""
import importlib.util
import os

import numpy as np
import pytest

from oracle import layer
from tests.rotations import random_rotation, wigner_d_blocks
from equivariant_gnn_message_gb300.inputs import make_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gen():
    spec = importlib.util.spec_from_file_location(
        "gen_tables", os.path.join(ROOT, "equivariant_gnn_message_gb300", "csrc", "gen_tables.py"))
    g = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(g)
    return g


def _blocks(l):
    return slice(l * l, (l + 1) * (l + 1))


def _aligned_layer(g, wl, W):
    """Receiver sums by the aligned-frame schedule; W[e, p, c]."""
    terms = g.aligned_terms()
    C = wl.channels
    out = np.zeros((wl.n_atoms, C, 16))
    for e in range(wl.n_edges):
        v = wl.vec[e].astype(np.float64)
        r = np.linalg.norm(v)
        x = wl.x[wl.src[e]].astype(np.float64)
        if r * r < 1e-30:
            continue  # not produced by the generator
        Q = g.frame_from_direction((v / r).tolist())
        D = g.wigner_real(Q)
        xr = x.copy()
        for l in (1, 2, 3):
            xr[:, _blocks(l)] = x[:, _blocks(l)] @ np.array(D[l])        # D^T x, row form
        mp = np.zeros((C, 16))
        for (p, k3, k1, kappa) in terms:
            mp[:, k3] += W[e, p] * kappa * xr[:, k1]
        m = mp.copy()
        for l in (1, 2, 3):
            m[:, _blocks(l)] = mp[:, _blocks(l)] @ np.array(D[l]).T       # D m'
        out[wl.dst[e]] += m
    return out


@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_aligned_schedule_equals_dense_layer(mode):
    g = _gen()
    wl = make_workload(n_atoms=24, cutoff=5.0, channels=3, weights=mode, storage="f32", seed=17)
    if mode == "shared":
        W = np.broadcast_to(wl.w.astype(np.float64)[None], (wl.n_edges, 34, 3))
        kw = dict(w=wl.w)
    else:
        W = (wl.R.astype(np.float64) @ wl.M.astype(np.float64)).reshape(wl.n_edges, 34, 3)
        kw = dict(R=wl.R, M=wl.M)
    got = _aligned_layer(g, wl, W)
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **kw)
    assert np.max(np.abs(got - want)) < 1e-10 * np.max(np.abs(want))


def test_generator_wigner_matches_fitted_blocks():
    g = _gen()
    for seed in range(4):
        Q = random_rotation(seed)
        Df = wigner_d_blocks(Q)
        Dg = g.wigner_real(Q.tolist())
        for l in (1, 2, 3):
            assert np.allclose(np.array(Dg[l]), Df[l], atol=1e-12)


def test_frame_is_a_rotation_taking_z_to_the_edge():
    g = _gen()
    rng = np.random.default_rng(3)
    dirs = np.concatenate([rng.standard_normal((50, 3)), [[0, 0, 1], [0, 0, -1], [1e-9, 0, -1]]])
    for n in dirs:
        n = n / np.linalg.norm(n)
        Q = np.array(g.frame_from_direction(n.tolist()))
        assert np.allclose(Q.T @ Q, np.eye(3), atol=1e-12)
        assert np.linalg.det(Q) > 0
        assert np.allclose(Q[:, 2], n, atol=1e-15)


def test_aligned_terms_selection_rule():
    """Eq. 13: per path each output m3 takes one input m1 (m1 = +m3 even,
    -m3 odd); 111 terms in all."""
    g = _gen()
    terms = g.aligned_terms()
    assert len(terms) == 111
    seen = set()
    for (p, k3, k1, kappa) in terms:
        assert (p, k3) not in seen
        seen.add((p, k3))
