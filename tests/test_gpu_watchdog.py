"""Failure reporting on a live GPU, without a fault: a bounded wait that
nothing completes gives up, the host reads its code, and the device keeps
working."""
import numpy as np
import pytest

from equivariant_gnn_message_gb300.inputs import make_workload
from oracle import layer
from tests.gpu_util import TOL, host, oracle_kw, rel_err, to_device, weights_kw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eq():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as m

    torch.cuda.set_device(0)
    return m


def test_expired_wait_is_reported_and_the_device_stays_usable(eq):
    import torch

    assert eq.eqmp_device_error() == 0
    eq.eqmp_watchdog_selftest(20)
    torch.cuda.synchronize()
    assert eq.eqmp_device_error() == 5          # read and cleared
    assert eq.eqmp_device_error() == 0
    wl = make_workload("tiny_64")
    d = to_device(wl)
    got = host(eq.eqmp_fused(d["vec"], d["x"], d["off"], d["src"], **weights_kw(d)))
    want = layer.message_pass(wl.vec, wl.x, wl.off, wl.src, **oracle_kw(wl))
    assert rel_err(got, want) <= TOL["f32"]
    assert eq.eqmp_device_error() == 0


def test_selftest_argument_range(eq):
    for bad in (0, -3, 5000):
        with pytest.raises(eq.EqmpError):
            eq.eqmp_watchdog_selftest(bad)
