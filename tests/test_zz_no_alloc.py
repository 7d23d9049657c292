"""The allocation-free backward entry point against the regular one.

eqmp_fused_backward_noalloc serves callers that cannot give the library
device memory (a plugin inside a framework that owns the memory pool, a
simulation loop that must not allocate every step).  Its scratch is a
static device array shared by all calls.  This test calls it through the C
ABI twice in a row (the second call starts from the first call's leftover
scratch) and compares every gradient with eqmp_fused_backward and with the
CPU oracle's gradients, within the parity tolerance of the GPU tests.  It
runs last so a failure here leaves the rest of the suite already run.
"""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import backward

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    scale = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / scale) if scale > 0 else float(np.max(np.abs(a)))


@pytest.mark.parametrize("mode,C,n_atoms", [("shared", 32, 400), ("shared", 64, 500), ("shared", 128, 600),
                                             ("radial", 8, 40)])
def test_noalloc_backward_matches_workspace_backward(mode, C, n_atoms):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as eq

    torch.cuda.set_device(0)
    wl = make_workload(n_atoms=n_atoms, cutoff=5.0, channels=C, weights=mode, storage="f32", seed=300 + C)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    so, se = eq.sender_view(wl.src, wl.n_atoms)
    need = ("x", "vec", "w") if mode == "shared" else ("x", "vec", "R", "M")
    kw = dict(w=t(wl.w), R=t(wl.R), M=t(wl.M), need=need)
    for call in range(2):
        g = torch.randn((wl.n_atoms, C, 16), device="cuda", generator=torch.Generator(device="cuda").manual_seed(call))
        args = (t(wl.vec), t(wl.x), t(wl.off), t(wl.src), t(wl.dst), t(so), t(se), g)
        ref = eq.eqmp_fused_backward(*args, **kw)
        got = eq.eqmp_fused_backward_noalloc(*args, **kw)
        torch.cuda.synchronize()
        okw = dict(w=wl.w) if mode == "shared" else dict(R=wl.R, M=wl.M)
        want = backward.layer_backward(wl.vec, wl.x, wl.off, wl.src, g.cpu().numpy(), **okw)
        for k in need:
            err = _rel(got[k], ref[k])
            assert err <= TOL, f"call {call}, grad {k}: rel err {err:.3e} against the workspace entry"
            err = _rel(got[k], torch.from_numpy(want[k]))
            assert err <= TOL, f"call {call}, grad {k}: rel err {err:.3e} against the oracle"
    assert eq.eqmp_device_error() == 0
    assert eq.load_library().eqmp_fused_backward_noalloc_max_bytes() == 8 << 20


def test_noalloc_rejects_radial_beyond_the_static_scratch():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as eq

    wl = make_workload("radial_1k_c32")  # E * 34 * 32 * 4 bytes > 8 MiB
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    so, se = eq.sender_view(wl.src, wl.n_atoms)
    g = torch.zeros((wl.n_atoms, 32, 16), device="cuda")
    with pytest.raises(eq.EqmpError) as ei:
        eq.eqmp_fused_backward_noalloc(t(wl.vec), t(wl.x), t(wl.off), t(wl.src), t(wl.dst), t(so), t(se), g,
                                       R=t(wl.R), M=t(wl.M), need=("vec",))
    assert ei.value.status == eq.EQMP_ERR_UNSUPPORTED
