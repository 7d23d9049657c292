"""The full-size oracle helper (tests/oracle_pool.py) against one oracle call.

The helper only cuts the receivers into ranges and runs the unchanged
oracle on each in spawned processes: on small graphs its forward result
must equal one call bit for bit, and its summed backward gradients one
call's to rounding.
"""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import backward, layer
from tests import oracle_pool


def test_forward_ranges_equal_one_call():
    for name, kw in (("tiny_64", {}), (None, dict(n_atoms=150, cutoff=5.0, channels=8, weights="radial",
                                                  storage="f32", seed=7))):
        wl = make_workload(name, **kw)
        want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src,
                                  **(dict(w=wl.w) if wl.w is not None else dict(R=wl.R, M=wl.M)))
        got = oracle_pool.message_pass_all(wl, workers=3)
        assert np.array_equal(got, want)


@pytest.mark.parametrize("mode", ["shared", "radial"])
def test_backward_ranges_sum_to_one_call(mode):
    wl = make_workload(n_atoms=150, cutoff=5.0, channels=8, weights=mode, storage="f32", seed=7)
    g = np.random.default_rng(0).standard_normal((wl.n_atoms, 8, 16)).astype(np.float32)
    kw = dict(w=wl.w) if wl.w is not None else dict(R=wl.R, M=wl.M)
    want = backward.layer_backward(wl.vec, wl.x, wl.off, wl.src, g, **kw)
    got = oracle_pool.layer_backward_all(wl, g, workers=3)
    assert sorted(got) == sorted(want)
    for k in want:
        assert got[k].shape == want[k].shape
        assert np.max(np.abs(got[k] - want[k])) <= 1e-12 * np.max(np.abs(want[k])), k
