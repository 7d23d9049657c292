"""Random rotations and real Wigner-D blocks fitted from harmonics (tests)."""
import numpy as np

from oracle import sh


def random_rotation(seed):
    """Haar-random proper rotation from a QR decomposition."""
    rng = np.random.default_rng(seed)
    q, r = np.linalg.qr(rng.standard_normal((3, 3)))
    q = q * np.sign(np.diag(r))[None, :]
    if np.linalg.det(q) < 0:
        q[:, 0] = -q[:, 0]
    return q


def wigner_d_blocks(Q, n_dirs=64, seed=123, l_max=3):
    """D_l(Q), l = 0..l_max, with Y_l(Q n) = D_l Y_l(n), fitted by least squares.

    Each block is checked to be orthogonal with determinant +1 before use.
    """
    rng = np.random.default_rng(seed)
    n = rng.standard_normal((max(n_dirs, 4 * (2 * l_max + 1)), 3))
    n /= np.linalg.norm(n, axis=1, keepdims=True)
    Y0, Y1 = sh.real_sh(n, l_max), sh.real_sh(n @ Q.T, l_max)
    blocks = []
    for l in range(l_max + 1):
        blk = slice(l * l, (l + 1) ** 2)
        # Y1[:, blk] = Y0[:, blk] @ D^T
        Dt, *_ = np.linalg.lstsq(Y0[:, blk], Y1[:, blk], rcond=None)
        D = Dt.T
        assert np.allclose(D @ D.T, np.eye(2 * l + 1), atol=1e-10)
        assert np.linalg.det(D) > 0
        blocks.append(D)
    return blocks


def rotate_features(x, blocks):
    """x[..., (l_max+1)^2] -> per-l-block D_l x."""
    out = np.empty_like(np.asarray(x, dtype=np.float64))
    for l, D in enumerate(blocks):
        blk = slice(l * l, (l + 1) ** 2)
        out[..., blk] = np.einsum("ab,...b->...a", D, x[..., blk])
    return out
