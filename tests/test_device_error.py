"""The device error path, made to happen on purpose without any fault: a
bounded wait on a barrier that nothing arrives on gives up, sets the device
status word and releases its tensor memory; the host reads and clears the
word, and the context stays usable for a forward checked against the oracle."""
import pytest
import torch

from higher_order_linear_gb300 import hla2
from tests._parity import TOL_TC_BF16, f64, oracle_forward, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def test_wait_runout_sets_status_and_context_survives():
    assert hla2.hla2_device_status() == 0  # nothing pending
    flag = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    hla2.hla2_selftest_wait_runout(flag, 20000)  # 20 ms
    assert hla2.hla2_device_status() == hla2.HLA2_ERR_DEVICE
    assert "wait" in hla2.hla2_last_error_detail()
    assert int(flag.item()) == 0  # the wait gave up
    assert hla2.hla2_device_status() == 0  # read and cleared
    # the same context runs a forward to the oracle's bound afterwards
    g = torch.Generator().manual_seed(3)
    q, k, v = ((torch.randn(1, 2, 300, 64, generator=g) / 8).to(torch.bfloat16) for _ in range(3))
    out = hla2.hla2_forward(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert hla2.hla2_device_status() == 0
    assert relerr(f64(out), oracle_forward(q, k, v)) < TOL_TC_BF16


def test_wait_runout_repeats():
    """Several run-outs in a row, each reported once."""
    flag = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    for _ in range(3):
        hla2.hla2_selftest_wait_runout(flag, 1000)
        assert hla2.hla2_device_status() == hla2.HLA2_ERR_DEVICE
        assert hla2.hla2_device_status() == 0
