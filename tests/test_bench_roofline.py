"""The bench's roofline arithmetic against hand-computed values (CPU only)."""
import pytest

import bench
from equivariant_gnn_message_gb300.inputs import make_workload


def test_shared_weights_pages():
    wl = make_workload("pages_1k_c32")
    flops, basis, extra = bench.layer_flops(wl, "forward", 3)
    assert flops == 2.0 * (256 * 32 * wl.n_edges + 767 * 32 * wl.n_atoms)
    nbytes = bench.compulsory_bytes(wl)
    assert nbytes == 2 * 1000 * 32 * 16 * 4 + 16 * wl.n_edges + 4 * 1001 + 4 * 34 * 32
    r = bench.roofline(flops, nbytes, 0.0174, 80.54784, 6793.1, "k", None, basis, extra)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(flops / 80.54784e12 / 17.4e-6)
    assert r["frac"] == pytest.approx(0.228, abs=0.001)


def test_radial_is_graded_on_the_aligned_schedule():
    wl = make_workload("radial_1k_c32")
    flops, basis, extra = bench.layer_flops(wl, "forward", 3)
    assert flops == 2.0 * 549 * 32 * wl.n_edges              # 2*83 rotations + 111 terms + 272 weights
    assert extra["flops_dense_basis"] == 2.0 * ((611 + 156 + 272) * 32 + 611) * wl.n_edges
    r = bench.roofline(flops, bench.compulsory_bytes(wl), 0.0377, 80.54784, 6793.1, "k", None, basis, extra)
    assert r["frac_dense_basis"] / r["frac"] == pytest.approx(extra["flops_dense_basis"] / flops)


def test_bound_follows_the_larger_time():
    r = bench.roofline(1e9, 1e12, 1.0, 80.0, 6800.0, "k", None, "b")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx((1e12 / 6800e9) / 1e-3)
    r = bench.roofline(1e12, 1e6, 1.0, 80.0, 6800.0, "k", None, "b")
    assert r["bound"] == "alu" and r["frac"] == pytest.approx((1e12 / 80e12) / 1e-3)


def test_degree_six_and_backward_counts():
    wl = make_workload("pages_1k_c32", l_max=6)
    flops, _, _ = bench.layer_flops(wl, "forward", 6)
    rot = sum((2 * l + 1) ** 2 for l in range(1, 7))
    assert flops == 2.0 * (2 * rot + 1036) * 32 * wl.n_edges
    wl = make_workload("pages_1k_c32")
    flops, _, _ = bench.layer_flops(wl, "backward", 3)
    assert flops == 2.0 * (3 * (256 * 32 * wl.n_edges + 767 * 32 * wl.n_atoms) + 48 * wl.n_edges)
