"""GPU forward on host buffers (hla2_forward_host through the C ABI): groups
of heads are copied in, computed and copied out as a pipeline.  Results are
compared with the fp64 oracle and with hla2_forward on device buffers."""
import pytest
import torch

from higher_order_linear_gb300 import hla2, workloads as W
from tests._parity import TOL_FP32_WALK, TOL_TC_BF16, f64, oracle_forward, relerr

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from higher_order_linear_gb300 import build
    build.build()


def inputs(B, H, T, d, dv, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, T, d, generator=g) / d ** 0.5
    k = torch.randn(B, H, T, d, generator=g) / d ** 0.5
    v = torch.randn(B, H, T, dv, generator=g) / d ** 0.5
    return q.to(dtype), k.to(dtype), v.to(dtype)


def run_host(q, k, v, heads_per_group=0):
    torch.cuda.set_device(0)
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    O = hla2.hla2_forward_host(qh, kh, vh, heads_per_group=heads_per_group)
    torch.cuda.current_stream().synchronize()
    assert hla2.hla2_device_status() == 0
    return O


@pytest.mark.parametrize("B,H,T,d,heads_per_group", [(1, 16, 2000, 128, 0), (2, 5, 700, 64, 3), (1, 4, 129, 64, 1),
                                                     (1, 6, 300, 128, 6), (3, 1, 1000, 64, 0)])
def test_host_forward_matches_oracle_and_device_forward(B, H, T, d, heads_per_group):
    q, k, v = inputs(B, H, T, d, d, torch.bfloat16, seed=B * 100 + H * 10 + T + d)
    got = run_host(q, k, v, heads_per_group)
    assert not got.is_cuda and got.shape == (B, H, T, d)
    ref = oracle_forward(q, k, v)
    assert relerr(f64(got), ref) < TOL_TC_BF16
    dev = hla2.hla2_forward(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert relerr(f64(got), f64(dev)) < TOL_TC_BF16


def test_host_forward_fp32_inputs():
    q, k, v = inputs(1, 3, 300, 32, 16, torch.float32, seed=5)
    got = run_host(q, k, v, 2)
    assert relerr(f64(got), oracle_forward(q, k, v)) < TOL_FP32_WALK


def test_host_forward_one_group_equals_device_forward_bit_for_bit():
    """With all heads in one group the host call runs exactly hla2_forward's
    launches on the same problem."""
    q, k, v = inputs(1, 8, 1500, 64, 64, torch.bfloat16, seed=9)
    got = run_host(q, k, v, heads_per_group=8)
    dev = hla2.hla2_forward(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(got, dev.cpu())


def test_host_forward_back_to_back_calls():
    """Calls share the copy streams and events: consecutive calls on new
    inputs give each call's own result."""
    w = W.WORKLOADS[1]
    outs, refs, pinned = [], [], []
    for seed in (1, 2, 3):
        q, k, v = W.make_inputs(w, seed=seed)
        qh, kh, vh = (x.pin_memory() for x in (q, k, v))
        pinned.append((qh, kh, vh))  # the copies read them until the stream is synchronised
        outs.append(hla2.hla2_forward_host(qh, kh, vh, heads_per_group=4))
        refs.append((q, k, v))
    torch.cuda.current_stream().synchronize()
    for O, (q, k, v) in zip(outs, refs):
        dev = hla2.hla2_forward(q.to(DEV), k.to(DEV), v.to(DEV))
        torch.cuda.synchronize()
        assert relerr(f64(O), f64(dev)) < TOL_TC_BF16
