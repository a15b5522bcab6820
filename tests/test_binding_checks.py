"""The Python binding checks its arguments before it touches the library or
the GPU: mismatched dtypes, wrong output shapes, dtypes or layouts, and
tensors on different devices raise ValueError, and nothing is launched
(CPU only: the checks fire before the first CUDA call)."""
import pytest
import torch

from higher_order_linear_gb300 import hla2


def _qkv(B=1, H=2, T=5, d=8, dv=8, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(0)
    mk = lambda n: torch.randn(B, H, T, n, generator=g).to(dtype)
    return mk(d), mk(d), mk(dv)


FORWARDS = [
    ("hla2_forward", lambda q, k, v, **kw: hla2.hla2_forward(q, k, v, **kw)),
    ("hla2_forward_noalloc", lambda q, k, v, **kw: hla2.hla2_forward_noalloc(q, k, v, **kw)),
    ("hla2_ahla_forward", lambda q, k, v, **kw: hla2.hla2_ahla_forward(q, k, v, **kw)),
    ("hla2_unmasked_forward", lambda q, k, v, **kw: hla2.hla2_unmasked_forward(q, k, v, **kw)),
    ("hla2_decay_forward", lambda q, k, v, **kw: hla2.hla2_decay_forward(q, k, v, 0.9, **kw)),
]


@pytest.mark.parametrize("name,fwd", FORWARDS)
def test_mixed_dtypes_rejected(name, fwd):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="share a dtype"):
        fwd(q, k.float(), v)
    with pytest.raises(ValueError, match="share a dtype"):
        fwd(q.float(), k.float(), v)


@pytest.mark.parametrize("name,fwd", FORWARDS)
def test_output_shape_dtype_layout_rejected(name, fwd):
    q, k, v = _qkv()
    B, H, T, _ = q.shape
    dv = v.shape[-1]
    for bad, what in ((torch.zeros(B, H, T - 1, dv), "shape"),
                      (torch.zeros(B, H, T, dv + 1), "shape"),
                      (torch.zeros(B, H, T, dv, dtype=torch.float64), "float32"),
                      (torch.zeros(B, H, dv, T).transpose(-1, -2), "contiguous")):
        before = bad.clone()
        with pytest.raises(ValueError, match=what):
            fwd(q, k, v, O=bad)
        assert torch.equal(bad, before)


@pytest.mark.parametrize("name,fwd", FORWARDS)
def test_inputs_on_different_devices_rejected(name, fwd):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="is on meta"):
        fwd(q, k.to("meta"), v)
    with pytest.raises(ValueError, match="is on meta"):
        fwd(q, k, v, O=torch.empty(q.shape[:3] + (v.shape[-1],), device="meta"))


def test_cpu_inputs_rejected_before_any_launch():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA tensor"):
        hla2.hla2_forward_noalloc(q, k, v)


@pytest.mark.parametrize("entry", ["hla2_step", "hla2_step_pform", "hla2_ahla_step", "hla2_unmasked_step"])
def test_step_argument_checks(entry):
    fn = getattr(hla2, entry)
    lens = {"hla2_step": hla2.record_len, "hla2_step_pform": hla2.pform_record_len,
            "hla2_ahla_step": hla2.ahla_state_len, "hla2_unmasked_step": hla2.unmasked_state_len}
    n, d, dv = 3, 8, 8
    state = torch.zeros(n, lens[entry](d, dv))
    q = torch.zeros(n, d)
    v = torch.zeros(n, dv)
    with pytest.raises(ValueError, match="state must hold"):
        fn(state[:-1], q, q, v)
    with pytest.raises(ValueError, match="o has shape"):
        fn(state, q, q, v, o=torch.zeros(n, dv + 1))
    with pytest.raises(ValueError, match="is on meta"):
        fn(state, q, q.to("meta"), v)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fn(state, q, q, v)
