"""eqmp_fused_staged (inputs and result in host memory, one C-ABI call per
step) against eqmp_fused on device memory (bit for bit) and the oracle."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import layer
from tests.gpu_util import TOL, oracle_kw, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eq():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as m

    torch.cuda.set_device(0)
    return m


def _pack(torch, wl):
    """The step's arrays in one pinned host block (256-byte aligned parts)
    and the same layout on the device; returns views into the device block."""
    parts = {"vec": wl.vec, "off": wl.off, "src": wl.src,
             "x": wl.x_bf16_bits.view(np.int16) if wl.storage == "bf16" else wl.x}
    for k in ("w", "R", "M"):
        if getattr(wl, k) is not None:
            parts[k] = getattr(wl, k)
    layout, n = {}, 0
    for k, a in parts.items():
        a = np.ascontiguousarray(a)
        layout[k] = (n, a)
        n = (n + a.nbytes + 255) // 256 * 256
    h = torch.zeros(n, dtype=torch.uint8).pin_memory()
    for k, (o, a) in layout.items():
        h.numpy()[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32, np.dtype(np.int16): torch.int16}
    views = {k: d[o:o + a.nbytes].view(tdt[a.dtype]).view(a.shape) for k, (o, a) in layout.items()}
    if wl.storage == "bf16":
        views["x"] = views["x"].view(torch.bfloat16)
    return h, d, views


@pytest.mark.parametrize("name", ["pages_1k_c32", "radial_1k_c32", "dense_10k_c128_bf16", "tiny_64"])
def test_staged_equals_device_call_and_oracle(eq, name):
    import torch

    wl = make_workload(name)
    h, d, v = _pack(torch, wl)
    kw = dict(w=v.get("w"), R=v.get("R"), M=v.get("M"))
    out = torch.empty((wl.n_atoms, wl.channels, 16), dtype=v["x"].dtype, device="cuda")
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    for _ in range(2):  # the second call starts from the first call's buffers
        h_out.fill_(float("nan"))
        eq.eqmp_fused_staged(h, d, v["vec"], v["x"], v["off"], v["src"], out, h_out, **kw)
        torch.cuda.synchronize()
        ref = eq.eqmp_fused(v["vec"], v["x"], v["off"], v["src"], **kw)
        torch.cuda.synchronize()
        assert torch.equal(h_out, ref.cpu())
    got = h_out.float().numpy().astype(np.float64)
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **oracle_kw(wl))
    assert rel_err(got, want) <= TOL[wl.storage]
    assert eq.eqmp_device_error() == 0


def test_prepared_staged_call_on_two_streams(eq):
    """prepare=True returns a call that repeats the step on the same
    buffers; two prepared calls on two streams, alternating, give the same
    bits as the one-off call."""
    import torch

    wl = make_workload("pages_1k_c32")
    sets = []
    for _ in range(2):
        h, d, v = _pack(torch, wl)
        out = torch.empty((wl.n_atoms, wl.channels, 16), dtype=v["x"].dtype, device="cuda")
        h_out = torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory()
        sets.append((h, d, v, out, h_out))
    h, d, v, out, h_out = sets[0]
    eq.eqmp_fused_staged(h, d, v["vec"], v["x"], v["off"], v["src"], out, h_out, w=v["w"])
    torch.cuda.synchronize()
    ref = h_out.clone()
    streams = [torch.cuda.Stream() for _ in range(2)]
    runs = [eq.eqmp_fused_staged(hh, dd, vv["vec"], vv["x"], vv["off"], vv["src"], oo, ho, w=vv["w"],
                                 stream=streams[b], prepare=True)
            for b, (hh, dd, vv, oo, ho) in enumerate(sets)]
    for i in range(6):
        runs[i % 2]()
    torch.cuda.synchronize()
    for b in range(2):
        assert sets[b][4].equal(ref)
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, w=wl.w)
    assert rel_err(ref.numpy().astype(np.float64), want) <= TOL["f32"]
    assert eq.eqmp_device_error() == 0


@pytest.mark.parametrize("name", ["pages_1k_c32", "radial_1k_c32"])
def test_plan_replays_the_staged_step(eq, name):
    """eqmp_plan_staged records the step once; launches on two streams (two
    plans over two buffer sets) give the one-off call's bits, and the plan
    follows new input contents.  Radial weights record the aligned-frame
    kernel's cluster launch."""
    import torch

    wl = make_workload(name)
    sets = []
    for _ in range(2):
        h, d, v = _pack(torch, wl)
        out = torch.empty((wl.n_atoms, wl.channels, 16), dtype=v["x"].dtype, device="cuda")
        h_out = torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory()
        sets.append((h, d, v, out, h_out))
    h, d, v, out, h_out = sets[0]
    def kw(vv):
        return dict(w=vv.get("w"), R=vv.get("R"), M=vv.get("M"))

    eq.eqmp_fused_staged(h, d, v["vec"], v["x"], v["off"], v["src"], out, h_out, **kw(v))
    torch.cuda.synchronize()
    ref = h_out.clone()
    plans = [eq.eqmp_plan_staged(hh, dd, vv["vec"], vv["x"], vv["off"], vv["src"], oo, ho, **kw(vv))
             for hh, dd, vv, oo, ho in sets]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for b in range(2):
        sets[b][4].fill_(float("nan"))
    for i in range(6):
        plans[i % 2].launch(streams[i % 2])
    torch.cuda.synchronize()
    for b in range(2):
        assert sets[b][4].equal(ref)
    # new features in the host block: the next launch copies and uses them
    h0 = sets[0][0]
    xo = v["x"].data_ptr() - d.data_ptr()
    nx = wl.x.nbytes
    h0.numpy()[xo:xo + nx] = (2.0 * wl.x).view(np.uint8).reshape(-1)
    plans[0].launch(streams[0])
    torch.cuda.synchronize()
    assert torch.allclose(sets[0][4], 2.0 * ref, rtol=1e-6, atol=1e-6)
    for p in plans:
        p.destroy()
    assert eq.eqmp_device_error() == 0
