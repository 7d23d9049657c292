"""Seeded synthetic workloads: random atom clouds, radius graphs, features.

This module generates inputs only; it holds none of the layer's arithmetic
(no harmonics, no CG, no tensor product).  Both the CUDA path and the CPU
oracle are fed the arrays it returns.

Recipe (one generator for every workload):
  * positions uniform in an open cube of side (N / 0.038)^(1/3) Angstrom
    (number density 0.038 / A^3, no periodic images);
  * directed edges for every ordered pair i != j closer than the cutoff,
    sender j -> receiver i, sorted by (receiver, sender); receiver i owns
    CSR rows off[i] .. off[i+1]-1;
  * edge vector vec_e = pos[src_e] - pos[dst_e] (receiver to sender), fp32;
  * node features x[N, C, 16] ~ N(0, 1), fp32, or rounded to bf16
    (round-to-nearest-even) for the bf16-storage workload;
  * shared per-path channel weights w[34, C] ~ N(0, std = 1/sqrt(34)), or,
    for the radial workload, M[8, 34*C] ~ N(0, std = 1/sqrt(8)) and
    R[E, 8] = Gaussian basis (8 centres linspace(0, 5, 8) A, sigma 0.5 A)
    times the cosine envelope 0.5 (cos(pi d / 5) + 1) for d < 5 A.
  Draw order from numpy.random.default_rng(seed): positions, x, then w or M.

The workloads mirror the sizes on the Batmobile blog (1000 atoms, 32
channels, about 20 neighbours, cutoff 4-6 A, 1000-5000 atoms per batch)
and E2Former-V2's dense regime (k about 30-100 neighbours, N ~ 1e4).

Atom order: draw order (spatially random, the hardest case for the row
gather), or, with order="morton", the same atoms and features renumbered
along the Morton (Z-order) curve of their cutoff-sized cells, the order a
cell-list neighbour builder leaves atoms in.  Renumbering is a permutation
of the input, applied before the graph is built.
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np

N_PATHS = 34
N_SH = 16
DENSITY = 0.038  # atoms / A^3

WORKLOADS = {
    # name: (n_atoms, cutoff A, channels, weight mode, storage, seed)
    "tiny_64":        dict(n_atoms=64, cutoff=5.0, channels=8, weights="shared", storage="f32", seed=1),
    "pages_1k_c32":   dict(n_atoms=1000, cutoff=5.0, channels=32, weights="shared", storage="f32", seed=2),
    "radial_1k_c32":  dict(n_atoms=1000, cutoff=5.0, channels=32, weights="radial", storage="f32", seed=3),
    "scale_100k_c64": dict(n_atoms=100_000, cutoff=5.0, channels=64, weights="shared", storage="f32", seed=4),
    "dense_10k_c128_bf16": dict(n_atoms=10_000, cutoff=7.0, channels=128, weights="shared", storage="bf16", seed=5),
    # a quarter of the scale workload (same density, cutoff and channels): the
    # size for multi-pass profiler captures of the C = 64 kernels (x 102 MB)
    "scale_25k_c64":  dict(n_atoms=25_000, cutoff=5.0, channels=64, weights="shared", storage="f32", seed=7),
    # the scale workload's atoms and features, renumbered in Morton order of their cells
    "scale_100k_c64_morton": dict(n_atoms=100_000, cutoff=5.0, channels=64, weights="shared", storage="f32", seed=4,
                                  order="morton"),
}


@dataclass
class Workload:
    name: str
    n_atoms: int
    channels: int
    storage: str               # "f32" or "bf16" (x and out)
    vec: np.ndarray            # [E, 3] float32
    src: np.ndarray            # [E] int32, CSR (receiver-sorted) order
    dst: np.ndarray            # [E] int32
    off: np.ndarray            # [N+1] int32, absolute edge offsets
    x: np.ndarray              # [N, C, 16] float32 (bf16-exact values when storage == "bf16")
    x_bf16_bits: Optional[np.ndarray]  # [N, C, 16] uint16 when storage == "bf16"
    w: Optional[np.ndarray]    # [34, C] float32
    R: Optional[np.ndarray]    # [E, 8] float32
    M: Optional[np.ndarray]    # [8, 34*C] float32
    pos: Optional[np.ndarray] = None  # [N, 3] float32 atom positions (rounded from the draw)
    cutoff: float = 0.0

    @property
    def n_edges(self) -> int:
        return int(self.src.shape[0])


def bf16_round_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def radius_graph(pos: np.ndarray, cutoff: float):
    """All ordered pairs closer than cutoff, sorted by (receiver, sender)."""
    from scipy.spatial import cKDTree

    pairs = cKDTree(pos).query_pairs(cutoff, output_type="ndarray")
    if pairs.size == 0:
        pairs = np.zeros((0, 2), dtype=np.int64)
    a, b = pairs[:, 0].astype(np.int64), pairs[:, 1].astype(np.int64)
    dst = np.concatenate([a, b])
    src = np.concatenate([b, a])
    order = np.lexsort((src, dst))
    return src[order], dst[order]


def csr_offsets(dst: np.ndarray, n: int) -> np.ndarray:
    return np.searchsorted(dst, np.arange(n + 1), side="left").astype(np.int32)


def radial_basis(d: np.ndarray, n_basis: int = 8, r_max: float = 5.0, sigma: float = 0.5) -> np.ndarray:
    mu = np.linspace(0.0, r_max, n_basis)
    g = np.exp(-((d[:, None] - mu[None, :]) ** 2) / (2.0 * sigma * sigma))
    env = np.where(d < r_max, 0.5 * (np.cos(np.pi * d / r_max) + 1.0), 0.0)
    return (g * env[:, None]).astype(np.float32)


def morton_order(pos: np.ndarray, cell: float) -> np.ndarray:
    """Permutation sorting atoms along the Morton curve of their cells
    (cell coordinates floor(p / cell), 21 bits per axis interleaved)."""
    c = np.floor(np.asarray(pos, np.float64) / cell).astype(np.int64)
    c -= c.min(axis=0) if len(c) else 0

    def spread(v):
        v = v.astype(np.uint64) & np.uint64(0x1FFFFF)
        out = np.zeros_like(v)
        for b in range(21):
            out |= ((v >> np.uint64(b)) & np.uint64(1)) << np.uint64(3 * b)
        return out

    key = spread(c[:, 0]) | (spread(c[:, 1]) << np.uint64(1)) | (spread(c[:, 2]) << np.uint64(2))
    return np.argsort(key, kind="stable")


def n_paths(l_max: int) -> int:
    """Number of (l1, l2, l3) with |l1-l2| <= l3 <= l1+l2, all <= l_max."""
    return sum(min(l_max, a + b) - abs(a - b) + 1 for a in range(l_max + 1) for b in range(l_max + 1))


def make_workload(name: str = None, *, n_atoms=None, cutoff=None, channels=None,
                  weights=None, storage=None, seed=None, l_max: int = 3) -> Workload:
    """Build a named workload, or a custom one from keyword overrides.

    l_max > 3 gives the higher-degree variant: x [N, C, (l_max+1)^2] and
    weights over all n_paths(l_max) paths (fp32 storage only).
    """
    spec = dict(WORKLOADS[name]) if name else {}
    for k, v in dict(n_atoms=n_atoms, cutoff=cutoff, channels=channels,
                     weights=weights, storage=storage, seed=seed).items():
        if v is not None:
            spec[k] = v
    n, C = int(spec["n_atoms"]), int(spec["channels"])
    rng = np.random.default_rng(spec["seed"])
    side = (n / DENSITY) ** (1.0 / 3.0)
    pos = rng.uniform(0.0, side, size=(n, 3))
    P = n_paths(l_max)
    x = rng.standard_normal((n, C, (l_max + 1) ** 2), dtype=np.float32)
    w = R = M = None
    if spec["weights"] == "shared":
        w = (rng.standard_normal((P, C)) / np.sqrt(P)).astype(np.float32)
    else:
        M = (rng.standard_normal((8, P * C)) / np.sqrt(8.0)).astype(np.float32)
    if spec.get("order", "draw") == "morton":
        perm = morton_order(pos, float(spec["cutoff"]))
        pos, x = pos[perm], x[perm]
    src, dst = radius_graph(pos, float(spec["cutoff"]))
    vec = (pos[src] - pos[dst]).astype(np.float32)
    if spec["weights"] != "shared":
        R = radial_basis(np.linalg.norm(pos[src] - pos[dst], axis=1))
    bits = None
    if spec["storage"] == "bf16":
        bits = bf16_round_bits(x)
        x = bf16_bits_to_f32(bits)
    return Workload(
        name=name or "custom", n_atoms=n, channels=C, storage=spec["storage"],
        vec=np.ascontiguousarray(vec), src=src.astype(np.int32), dst=dst.astype(np.int32),
        off=csr_offsets(dst, n), x=np.ascontiguousarray(x), x_bf16_bits=bits,
        w=w, R=R, M=M, pos=pos.astype(np.float32), cutoff=float(spec["cutoff"]))
