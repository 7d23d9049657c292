"""The C-ABI library builds, loads and exports every symbol include/eqmp.h
declares (CPU only: host-side functions only, no kernel launches)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "eqmp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(eqmp_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as eq

    return eq.load_library()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ("eqmp_sh", "eqmp_tp_scatter", "eqmp_fused", "eqmp_num_paths", "eqmp_path_table",
                 "eqmp_status_string", "eqmp_validate_graph", "eqmp_device_error"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_host_only_functions(lib):
    import equivariant_gnn_message_gb300 as eq
    from oracle import cg

    assert eq.eqmp_num_paths() == 34
    assert eq.eqmp_path_table() == cg.paths()
    assert eq.eqmp_status_string(0) == "ok"
    assert "unsupported" in eq.eqmp_status_string(2)
    assert eq.eqmp_status_string(99) == "unknown status"
    assert lib.eqmp_path_table(None) == eq.EQMP_ERR_INVALID_ARG


def test_fp32_probe_rejects_bad_arguments_before_any_launch(lib):
    """The probe's argument checks come before any CUDA call (no GPU needed)."""
    import equivariant_gnn_message_gb300 as eq

    flops = ctypes.c_double(-1.0)
    out = ctypes.c_void_p(16)  # never dereferenced: every call below fails its checks first
    for iters, bps, o, f in ((0, 4, out, ctypes.byref(flops)), (64, 0, out, ctypes.byref(flops)),
                             (64, 9, out, ctypes.byref(flops)), (64, 4, None, ctypes.byref(flops)),
                             (64, 4, out, None)):
        assert lib.eqmp_fp32_peak_probe(iters, bps, o, f, None) == eq.EQMP_ERR_INVALID_ARG
    assert flops.value == -1.0


def test_product_path_has_no_oracle_dependency():
    """The package and its sources never import or mention the oracle."""
    pkg = os.path.join(ROOT, "equivariant_gnn_message_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, re.M), f
                assert "oracle." not in text, f


def test_generated_tables_match_oracle():
    """The build-time CG generator (independent method) and the oracle agree."""
    import importlib.util

    import numpy as np

    from oracle import cg, sh

    spec = importlib.util.spec_from_file_location(
        "gen_tables", os.path.join(ROOT, "equivariant_gnn_message_gb300", "csrc", "gen_tables.py"))
    g = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(g)
    _, paths, terms = g.render()
    assert paths == cg.paths()
    assert len(terms) == 611
    for (l1, l2, l3, blk) in cg.real_cg_tables():
        ent = g.real_cg(l1, l2, l3)
        dense = np.zeros_like(blk)
        for (m3, m1, m2), v in ent.items():
            dense[m3 + l3, m1 + l1, m2 + l2] = v
        assert np.max(np.abs(dense - blk)) < 1e-12
    n = np.random.default_rng(0).standard_normal((20, 3))
    n /= np.linalg.norm(n, axis=1, keepdims=True)
    Y = sh.real_sh(n)
    shc = g.sh_constants()
    for l in range(4):
        for m in range(l + 1):
            poly = np.polynomial.polynomial.polyval(n[:, 2], shc[(l, m)])
            pw = (n[:, 0] + 1j * n[:, 1]) ** m
            assert np.allclose(poly * pw.real, Y[:, l * l + l + m], atol=1e-14)
            if m:
                assert np.allclose(poly * pw.imag, Y[:, l * l + l - m], atol=1e-14)


@pytest.mark.parametrize("entry", ["eqmp_fused_backward", "eqmp_fused_backward_noalloc"])
def test_backward_wrappers_reject_a_wrong_dtype_before_any_call(lib, entry):
    """A float64 x (or int64 index array) never reaches the C entry point as
    a raw pointer: the binding raises TypeError first (no GPU needed)."""
    import torch

    import equivariant_gnn_message_gb300 as eq

    f32, i32 = torch.float32, torch.int32
    args = dict(vec=torch.zeros(6, 3, dtype=f32), x=torch.zeros(3, 8, 16, dtype=f32),
                row_offsets=torch.zeros(4, dtype=i32), src=torch.zeros(6, dtype=i32),
                dst=torch.zeros(6, dtype=i32), send_offsets=torch.zeros(4, dtype=i32),
                send_edges=torch.zeros(6, dtype=i32), grad_out=torch.zeros(3, 8, 16, dtype=f32))
    fn = getattr(eq, entry)
    for name, bad in (("x", torch.zeros(3, 8, 16, dtype=torch.float64)),
                      ("src", torch.zeros(6, dtype=torch.int64)),
                      ("grad_out", torch.zeros(3, 8, 16, dtype=torch.float64))):
        kw = dict(args, **{name: bad})
        with pytest.raises(TypeError, match=name):
            fn(**kw, w=torch.zeros(34, 8, dtype=f32))
    with pytest.raises(ValueError, match="CUDA"):  # right dtypes, host memory
        fn(**args, w=torch.zeros(34, 8, dtype=f32))


def test_staged_entry_rejects_missing_blocks_before_any_copy(lib):
    """eqmp_fused_staged checks its host/device blocks and the output size
    before queueing anything (no GPU needed: every call below fails first)."""
    import equivariant_gnn_message_gb300 as eq

    d = ctypes.c_void_p(256)  # never dereferenced
    w = eq.Weights(d, None, None, 0)
    layer = (d, d, 8, eq.EQMP_F32, d, d, 4, 8, 8, w, d, eq.EQMP_F32)
    assert lib.eqmp_fused_staged(None, d, 16, *layer, d, 16, None) == eq.EQMP_ERR_INVALID_ARG   # no h_in
    assert lib.eqmp_fused_staged(d, None, 16, *layer, d, 16, None) == eq.EQMP_ERR_INVALID_ARG   # no d_in
    assert lib.eqmp_fused_staged(d, d, 16, *layer, None, 16, None) == eq.EQMP_ERR_INVALID_ARG   # no h_out
    # out holds 4 x 8 x 16 floats = 2048 bytes
    assert lib.eqmp_fused_staged(d, d, 16, *layer, d, 2049, None) == eq.EQMP_ERR_INVALID_ARG
