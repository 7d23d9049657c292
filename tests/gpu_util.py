"""Helpers for the GPU parity tests: upload a workload, compare with the oracle."""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_device(wl, dev="cuda"):
    import torch

    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = dict(vec=t(wl.vec), off=t(wl.off), src=t(wl.src), w=t(wl.w), R=t(wl.R), M=t(wl.M))
    if wl.storage == "bf16":
        d["x"] = torch.from_numpy(wl.x_bf16_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        d["x"] = t(wl.x)
    return d


def weights_kw(d):
    return dict(w=d["w"]) if d["w"] is not None else dict(R=d["R"], M=d["M"])


def oracle_kw(wl):
    return dict(w=wl.w) if wl.w is not None else dict(R=wl.R, M=wl.M)


def rel_err(got, want):
    got = np.asarray(got, dtype=np.float64)
    scale = np.max(np.abs(want)) if want.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - want)) / scale)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)
