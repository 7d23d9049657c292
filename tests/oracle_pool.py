"""The oracle over a whole full-size workload on all host cores (test helper).

Receivers are cut into contiguous ranges balanced on edges; spawned worker
processes (safe after the parent has used the GPU) each run the unchanged
oracle (``oracle.layer.message_pass``, ``oracle.backward.layer_backward``)
on their ranges.  Inputs and the output are memory-mapped ``.npy`` files in
a temporary directory, so no worker receives a copy of the feature array
and every output row is written by exactly one worker.  The split only
bounds the wall time: each output element is the oracle's own value for
its receiver (forward), or the sum over ranges of the oracle's per-range
gradients (backward: the gradient of a sum over receivers is the sum of
the gradients of its parts).
"""
import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

CHUNK_EDGES = 1024  # the oracle's memory-bounding group size (cache-friendly)


def _ranges(off, parts):
    off = np.asarray(off, dtype=np.int64)
    n = len(off) - 1
    cost = (off - off[0]) + 4 * np.arange(n + 1)
    cuts = [0] + [int(np.searchsorted(cost, cost[-1] * k / parts)) for k in range(1, parts)] + [n]
    cuts = np.maximum.accumulate(cuts)
    return [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


class _Files:
    def __init__(self, arrays):
        self.dir = tempfile.mkdtemp(prefix="eqmp_oracle_")
        self.paths = {}
        for k, a in arrays.items():
            if a is None:
                self.paths[k] = None
                continue
            p = os.path.join(self.dir, f"{k}.npy")
            np.save(p, np.ascontiguousarray(a))
            self.paths[k] = p

    def out(self, name, shape):
        p = os.path.join(self.dir, f"{name}.npy")
        np.lib.format.open_memmap(p, mode="w+", dtype=np.float64, shape=tuple(shape)).flush()
        return p

    def close(self):
        shutil.rmtree(self.dir, ignore_errors=True)


def _load(paths):
    return {k: (None if p is None else np.load(p, mmap_mode="r")) for k, p in paths.items()}


def _forward_part(args):
    paths, out_path, a, b = args
    from oracle import layer

    d = _load(paths)
    kw = dict(w=d["w"]) if d["w"] is not None else dict(R=d["R"], M=d["M"])
    res = layer.message_pass(d["vec"], d["x"], d["off"], d["src"], receivers=np.arange(a, b),
                             chunk_edges=CHUNK_EDGES, **kw)
    out = np.load(out_path, mmap_mode="r+")
    out[a:b] = res
    out.flush()
    return b - a


def _backward_part(args):
    paths, a, b = args
    from oracle import backward

    d = _load(paths)
    kw = dict(w=d["w"]) if d["w"] is not None else dict(R=d["R"], M=d["M"])
    off = np.asarray(d["off"][a:b + 1], dtype=np.int64)
    g = backward.layer_backward(d["vec"], d["x"], off, d["src"], np.asarray(d["g"][a:b]), **kw)
    e0, e1 = int(off[0]), int(off[-1])
    # rows of R and vec belong to this range's edges; x, w, M are partial sums
    part = {k: v for k, v in g.items() if k in ("x", "w", "M")}
    for k in ("R", "vec"):
        if k in g:
            part[k] = (e0, np.asarray(g[k][e0:e1]))
    return part


def _pool(workers):
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        return mp.get_context("spawn").Pool(workers)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _workers(workers):
    return max(1, int(workers or os.cpu_count() or 1))


def message_pass_all(wl, workers=None):
    """oracle.layer.message_pass over every receiver of wl (float64 [N, C, 16])."""
    n = _workers(workers)
    files = _Files(dict(vec=wl.vec, x=wl.x, off=wl.off, src=wl.src, w=wl.w, R=wl.R, M=wl.M))
    try:
        out_path = files.out("out", (wl.n_atoms, wl.channels, wl.x.shape[2]))
        jobs = [(files.paths, out_path, a, b) for a, b in _ranges(wl.off, 4 * n)]
        with _pool(n) as pool:
            done = sum(pool.map(_forward_part, jobs, chunksize=1))
        assert done == wl.n_atoms
        return np.array(np.load(out_path, mmap_mode="r"))
    finally:
        files.close()


def layer_backward_all(wl, g, workers=None):
    """oracle.backward.layer_backward over the whole graph of wl, evaluated
    per receiver range and summed (dict of float64 gradients)."""
    n = _workers(workers)
    files = _Files(dict(vec=wl.vec, x=wl.x, off=wl.off, src=wl.src, w=wl.w, R=wl.R, M=wl.M, g=g))
    try:
        jobs = [(files.paths, a, b) for a, b in _ranges(wl.off, 4 * n)]
        with _pool(n) as pool:
            parts = pool.map(_backward_part, jobs, chunksize=1)
    finally:
        files.close()
    E = wl.n_edges
    out = {}
    for part in parts:  # fixed order: receiver ranges ascending
        for k, v in part.items():
            if k in ("R", "vec"):
                e0, rows = v
                if k not in out:
                    out[k] = np.zeros((E, rows.shape[1]))
                out[k][e0:e0 + len(rows)] = rows
            else:
                out[k] = v if k not in out else out[k] + v
    return out
