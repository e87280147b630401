"""The binding runs each call on the device its tensors live on.

The library launches on the current CUDA device, so the binding checks that
every tensor of a call is on one device and makes that device current around
the call (with that device's current stream as the default).
"""

import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, swiglu_inputs, swish_inputs

from ._parity import assert_all, compare, to_f64


def test_device_of_refuses_mixed_devices():
    from swiglu_ffn_backward_gb300 import _binding as b
    a = torch.empty(4)
    m = torch.empty(4, device="meta")
    assert b._device_of(a, None, a) == a.device
    assert b._device_of(None, None) is None
    with pytest.raises(ValueError, match="one device"):
        b._device_of(a, m)


two_gpus = pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                              reason="needs two visible GPUs")


@pytest.mark.gpu
@two_gpus
def test_tensors_on_a_non_current_device():
    import swiglu_ffn_backward_gb300 as swg
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 1)
    grad, x = swish_inputs(4099, torch.bfloat16, device=dev, seed=3)
    gx = swg.swish_grad(grad, x, 1.702)
    assert gx.device == dev
    inp = swiglu_inputs(SWIGLU_CONFIGS["tiny"][0], device=dev)
    out = swg.swiglu_bwd(**inp, fused=True)
    with torch.cuda.device(dev):
        swg.swg_check()
    assert torch.cuda.current_device() == 0
    ref = oracle.swish_grad(to_f64(grad), to_f64(x), 1.702)
    h = {k: to_f64(v) for k, v in inp.items()}
    rdg, rdfc, _, _ = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    assert_all([compare("grad_x", gx, ref), compare("dg", out["dg"], rdg), compare("dfc", out["dfc"], rdfc)])


@pytest.mark.gpu
@two_gpus
def test_mixed_devices_are_refused():
    import swiglu_ffn_backward_gb300 as swg
    grad, x = swish_inputs(64, torch.float32, device="cuda:0", seed=3)
    with pytest.raises(ValueError):
        swg.swish_grad(grad, x.to("cuda:1"), 1.0)
