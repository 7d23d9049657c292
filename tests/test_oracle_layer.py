"""Pins for the oracle's tensor product + receiver sum (CPU only)."""
import itertools
from math import sqrt

import numpy as np
import pytest

from oracle import cg, layer, sh
from tests.rotations import random_rotation, rotate_features, wigner_d_blocks
from equivariant_gnn_message_gb300.inputs import make_workload, radial_basis


def _three_atoms(seed, C=3):
    rng = np.random.default_rng(seed)
    pos = rng.uniform(-2, 2, (3, 3))
    pairs = [(i, j) for i in range(3) for j in range(3) if i != j]  # (receiver, sender)
    dst = np.array([p[0] for p in pairs])
    src = np.array([p[1] for p in pairs])
    vec = pos[src] - pos[dst]
    off = np.searchsorted(dst, np.arange(4))
    x = rng.standard_normal((3, C, 16))
    w = rng.standard_normal((34, C))
    R = rng.standard_normal((6, 8))
    M = rng.standard_normal((8, 34 * C))
    return vec, src, dst, off, x, w, R, M


def _brute_force(vec, src, dst, x, n_recv, w=None, R=None, M=None):
    """Nested loops straight from the formula, one scalar at a time."""
    C = x.shape[1]
    out = np.zeros((n_recv, C, 16))
    tables = cg.real_cg_tables()
    for e in range(len(src)):
        Y = sh.real_sh(vec[e:e + 1])[0]
        for p, (l1, l2, l3, blk) in enumerate(tables):
            for c in range(C):
                W = w[p, c] if w is not None else sum(R[e, k] * M[k, p * C + c] for k in range(8))
                for m3, m1, m2 in itertools.product(range(-l3, l3 + 1), range(-l1, l1 + 1), range(-l2, l2 + 1)):
                    coef = blk[m3 + l3, m1 + l1, m2 + l2]
                    if coef == 0.0:
                        continue
                    out[dst[e], c, sh.sh_index(l3, m3)] += (
                        W * coef * x[src[e], c, sh.sh_index(l1, m1)] * Y[sh.sh_index(l2, m2)])
    return out


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_brute_force_three_atoms(seed, mode):
    vec, src, dst, off, x, w, R, M = _three_atoms(seed)
    kw = dict(w=w) if mode == "shared" else dict(R=R, M=M)
    got = layer.message_pass(vec, x, off, src, **kw)
    want = _brute_force(vec, src, dst, x, 3, **kw)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_scalar_features_give_weighted_harmonics():
    """x only in l1 = 0: out[i,c,(l,m)] = sum_e w[(0,l,l),c] x0 Y_e[(l,m)]."""
    vec, src, dst, off, x, w, R, M = _three_atoms(3)
    x[:, :, 1:] = 0.0
    got = layer.message_pass(vec, x, off, src, w=w)
    Y = sh.real_sh(vec)
    pidx = {p: i for i, p in enumerate(cg.paths())}
    want = np.zeros_like(got)
    for e in range(len(src)):
        for l in range(4):
            for m in range(-l, l + 1):
                k = sh.sh_index(l, m)
                want[dst[e], :, k] += w[pidx[(0, l, l)]] * x[src[e], :, 0] * Y[e, k]
    assert np.allclose(got, want, atol=1e-13)


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_rotation_equivariance(seed, mode):
    """out(Q vec, D x) = D out(vec, x), D fitted from the harmonics."""
    wl = make_workload(n_atoms=40, cutoff=5.0, channels=4, weights=mode, storage="f32", seed=10 + seed)
    kw = dict(w=wl.w) if mode == "shared" else dict(R=wl.R, M=wl.M)
    Q = random_rotation(100 + seed)
    D = wigner_d_blocks(Q)
    base = layer.message_pass(wl.vec.astype(np.float64), wl.x, wl.off, wl.src, **kw)
    rot = layer.message_pass(wl.vec.astype(np.float64) @ Q.T, rotate_features(wl.x, D),
                             wl.off, wl.src, **kw)
    assert np.max(np.abs(rot - rotate_features(base, D))) < 1e-11 * max(1.0, np.max(np.abs(base)))


def test_linearity_and_radial_equals_shared_when_constant():
    wl = make_workload(n_atoms=30, cutoff=5.0, channels=3, weights="radial", storage="f32", seed=4)
    # R constant 1 in slot 0, M[0] = w  ->  W = w
    R = np.zeros_like(wl.R)
    R[:, 0] = 1.0
    w = np.random.default_rng(0).standard_normal((34, 3))
    M = np.zeros((8, 34 * 3))
    M[0] = w.reshape(-1)
    a = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, R=R, M=M)
    b = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=w)
    assert np.allclose(a, b, atol=1e-13)
    c = layer.message_pass(wl.vec, 2.0 * wl.x, wl.off, wl.src, w=w)
    assert np.allclose(c, 2.0 * b, atol=1e-12)


def test_receiver_subsets_and_empty_receivers():
    wl = make_workload(n_atoms=50, cutoff=4.0, channels=2, weights="shared", storage="f32", seed=6)
    full = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=wl.w)
    sub = np.array([3, 17, 0, 49])
    part = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=wl.w, receivers=sub)
    assert np.allclose(part, full[sub], rtol=0, atol=1e-13)
    # small chunks give the same sums
    chunked = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=wl.w, chunk_edges=7)
    assert np.allclose(chunked, full, atol=1e-13)
    deg = np.diff(wl.off)
    assert np.all(full[deg == 0] == 0.0)
    # a graph with no edges at all
    z = layer.message_pass(np.zeros((0, 3)), wl.x, np.zeros(51, np.int64), np.zeros(0, np.int64), w=wl.w)
    assert z.shape == (50, 2, 16) and np.all(z == 0.0)


def test_planted_dropped_term_fails_brute_force(monkeypatch):
    """Zeroing one CG entry of one path makes the layer disagree with the
    independent brute force computed from the intact tables."""
    vec, src, dst, off, x, w, R, M = _three_atoms(5)
    want = _brute_force(vec, src, dst, x, 3, w=w)
    tables = cg.real_cg_tables()
    l1, l2, l3, blk = tables[23]
    bad = blk.copy()
    idx = np.argwhere(bad != 0)[0]
    bad[tuple(idx)] = 0.0
    planted = list(tables)
    planted[23] = (l1, l2, l3, bad)
    monkeypatch.setattr(cg, "real_cg_tables", lambda l_max=3: planted)
    got = layer.message_pass(vec, x, off, src, w=w)
    assert not np.allclose(got, want, atol=1e-9)


def test_radial_basis_recipe_values():
    d = np.array([0.0, 2.5, 5.0, 6.0])
    R = radial_basis(d)
    assert R.shape == (4, 8)
    assert abs(R[0, 0] - 1.0) < 1e-7                     # d = mu_0 = 0, envelope 1
    assert np.all(R[2:] == 0.0)                          # beyond the cutoff
    mu = np.linspace(0, 5, 8)
    env = 0.5 * (np.cos(np.pi * 2.5 / 5) + 1)
    assert np.allclose(R[1], np.exp(-(2.5 - mu) ** 2 / 0.5) * env, atol=1e-7)
