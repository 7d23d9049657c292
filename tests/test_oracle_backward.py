"""Pins for the oracle's gradients: central finite differences of the
(separately pinned) forward oracle, and rotation behaviour (CPU only)."""
import numpy as np
import pytest

from oracle import backward, layer, sh
from tests.rotations import random_rotation, rotate_features, wigner_d_blocks


def _graph(seed, n=4, C=2):
    rng = np.random.default_rng(seed)
    pos = rng.uniform(-1.5, 1.5, (n, 3))
    pairs = [(i, j) for i in range(n) for j in range(n) if i != j and (i + j) % 3 != 0]
    pairs.sort()
    dst = np.array([p[0] for p in pairs])
    src = np.array([p[1] for p in pairs])
    off = np.searchsorted(dst, np.arange(n + 1))
    vec = pos[src] - pos[dst]
    x = rng.standard_normal((n, C, 16))
    w = rng.standard_normal((34, C))
    R = rng.standard_normal((len(src), 8))
    M = rng.standard_normal((8, 34 * C))
    g = rng.standard_normal((n, C, 16))
    return vec, x, off, src, w, R, M, g


def _loss(vec, x, off, src, g, **kw):
    return float(np.sum(g * layer.message_pass(vec, x, off, src, **kw)))


def _fd(f, a, h=1e-6):
    a = np.array(a, dtype=np.float64)
    grad = np.zeros_like(a)
    it = np.nditer(a, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = a[idx]
        a[idx] = old + h
        fp = f(a)
        a[idx] = old - h
        fm = f(a)
        a[idx] = old
        grad[idx] = (fp - fm) / (2 * h)
    return grad


def test_sh_jacobian_matches_finite_differences():
    v = np.random.default_rng(0).standard_normal((7, 3)) * np.array([[1.0], [2.0], [0.5], [3.0], [1.0], [0.2], [4.0]])
    J = backward.sh_jacobian(v)
    for e in range(len(v)):
        for b in range(3):
            d = np.zeros(3)
            d[b] = 1e-6
            col = (sh.real_sh((v[e] + d)[None])[0] - sh.real_sh((v[e] - d)[None])[0]) / 2e-6
            assert np.allclose(J[e, :, b], col, atol=1e-8)
    # scale invariance of Y: radial derivative vanishes
    assert np.allclose(np.einsum("ekb,eb->ek", J, v), 0.0, atol=1e-12)


@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_gradients_match_finite_differences(mode):
    vec, x, off, src, w, R, M, g = _graph(1)
    kw = dict(w=w) if mode == "shared" else dict(R=R, M=M)
    got = backward.layer_backward(vec, x, off, src, g, **kw)
    fx = _fd(lambda a: _loss(vec, a, off, src, g, **kw), x)
    assert np.allclose(got["x"], fx, atol=1e-6)
    fv = _fd(lambda a: _loss(a, x, off, src, g, **kw), vec)
    assert np.allclose(got["vec"], fv, atol=1e-6)
    if mode == "shared":
        fw = _fd(lambda a: _loss(vec, x, off, src, g, w=a), w)
        assert np.allclose(got["w"], fw, atol=1e-6)
    else:
        fR = _fd(lambda a: _loss(vec, x, off, src, g, R=a, M=M), R)
        assert np.allclose(got["R"], fR, atol=1e-6)
        fM = _fd(lambda a: _loss(vec, x, off, src, g, R=R, M=a), M)
        assert np.allclose(got["M"], fM, atol=1e-6)


def test_force_gradient_rotates_as_a_vector():
    """dL/dvec(Q v, D x, D g) = Q dL/dvec(v, x, g); dL/dx rotates like x."""
    vec, x, off, src, w, R, M, g = _graph(2, n=5, C=3)
    Q = random_rotation(7)
    D = wigner_d_blocks(Q)
    a = backward.layer_backward(vec, x, off, src, g, w=w)
    b = backward.layer_backward(vec @ Q.T, rotate_features(x, D), off, src, rotate_features(g, D), w=w)
    assert np.allclose(b["vec"], a["vec"] @ Q.T, atol=1e-10)
    assert np.allclose(b["x"], rotate_features(a["x"], D), atol=1e-10)
    assert np.allclose(b["w"], a["w"], atol=1e-10)


def test_planted_sign_error_fails_fd():
    """A sign slip planted in the Jacobian is caught by finite differences."""
    vec, x, off, src, w, R, M, g = _graph(3)
    good = backward.layer_backward(vec, x, off, src, g, w=w)["vec"]
    fv = _fd(lambda a: _loss(a, x, off, src, g, w=w), vec)
    assert np.allclose(good, fv, atol=1e-6)
    assert not np.allclose(-good, fv, atol=1e-6)
