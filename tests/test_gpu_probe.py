"""The FP32 throughput probe on a live GPU: it reports the flop count of the
launch it made, runs to completion, and leaves its output word alone (the
sums never reach the guard value)."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eq():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import equivariant_gnn_message_gb300 as m

    torch.cuda.set_device(0)
    return m


@pytest.mark.parametrize("blocks_per_sm", [1, 4])
def test_probe_flop_count_and_output(eq, blocks_per_sm):
    import torch

    out = torch.zeros(1, device="cuda")
    iters = 256
    flops = eq.eqmp_fp32_peak_probe(iters, out, blocks_per_sm=blocks_per_sm)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert flops == sms * blocks_per_sm * 256 * 32 * iters
    assert out.item() == 0.0
    assert eq.eqmp_device_error() == 0


def test_probe_argument_errors(eq):
    import torch

    out = torch.zeros(1, device="cuda")
    for iters, bps in ((0, 4), (16, 0), (16, 9)):
        with pytest.raises(eq.EqmpError):
            eq.eqmp_fp32_peak_probe(iters, out, blocks_per_sm=bps)
