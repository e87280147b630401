"""SwishGrad through the C ABI vs the fp64 oracle (GPU)."""

import numpy as np
import pytest
import torch

import oracle
from synth import SWISH_CONFIG, swish_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _check(grad, x, scale, out):
    ref = oracle.swish_grad(to_f64(grad), to_f64(x), 1.0 if scale is None else scale)
    return compare("grad_x", out, ref, dtype=DT[grad.dtype])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
@pytest.mark.parametrize("scale", SWISH_CONFIG["scales"])
@pytest.mark.parametrize("n", SWISH_CONFIG["n"])
def test_swish_grad_full_size(n, scale, dtype):
    grad, x = swish_inputs(n, dtype, device="cuda", seed=SWISH_CONFIG["seed"])
    out = _swg().swish_grad(grad, x, scale)
    torch.cuda.synchronize()
    assert_all([_check(grad, x, scale, out)])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 31, 1000003])
def test_swish_grad_small_and_ragged(n, dtype):
    grad, x = swish_inputs(n, dtype, device="cuda", seed=5)
    out = _swg().swish_grad(grad, x, 1.702)
    torch.cuda.synchronize()
    assert_all([_check(grad, x, 1.702, out)])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
@pytest.mark.parametrize("offsets", [(1, 1, 1), (1, 2, 3), (0, 3, 5), (3, 3, 0)])
def test_swish_grad_unaligned(offsets, dtype):
    n = 100003
    g0, x0 = swish_inputs(n + 8, dtype, device="cuda", seed=6)
    o0 = torch.empty(n + 8, dtype=dtype, device="cuda")
    a, b, c = offsets
    grad, x, out = g0[a:a + n], x0[b:b + n], o0[c:c + n]
    _swg().swish_grad(grad, x, 1.0, grad_x=out)
    torch.cuda.synchronize()
    assert_all([_check(grad, x, 1.0, out)])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
def test_swish_grad_in_place_and_default_beta(dtype):
    grad, x = swish_inputs(4099, dtype, device="cuda", seed=7)
    g_copy, x_copy = grad.clone(), x.clone()
    _swg().swish_grad(grad, x, None, grad_x=grad)  # alias grad, beta NULL -> 1.0
    torch.cuda.synchronize()
    assert_all([_check(g_copy, x_copy, None, grad)])
    grad2, x2 = swish_inputs(4099, dtype, device="cuda", seed=8)
    g2, x2c = grad2.clone(), x2.clone()
    _swg().swish_grad(grad2, x2, 1.702, grad_x=x2)  # alias x
    torch.cuda.synchronize()
    assert_all([_check(g2, x2c, 1.702, x2)])


def test_swish_grad_special_values():
    swg = _swg()
    for dtype in SWISH_CONFIG["dtypes"]:
        grad = torch.randn(4096, device="cuda").to(dtype)
        # x = 0 or beta = 0: exactly grad / 2 in every dtype
        out = swg.swish_grad(grad, torch.zeros_like(grad), 1.702)
        assert torch.equal(out, (grad.float() / 2).to(dtype))
        out = swg.swish_grad(grad, torch.randn(4096, device="cuda").to(dtype), 0.0)
        assert torch.equal(out, (grad.float() / 2).to(dtype))
        # saturation: x -> +large gives grad, x -> -large gives 0
        big = torch.full_like(grad, 1e4 if dtype != torch.float16 else 6e4)
        assert torch.equal(swg.swish_grad(grad, big, 1.0), grad)
        assert torch.count_nonzero(swg.swish_grad(grad, -big, 1.0)) == 0


def test_swish_grad_empty():
    swg = _swg()
    e = torch.empty(0, device="cuda")
    out = swg.swish_grad(e, e, 1.0)
    assert out.numel() == 0


def test_swish_grad_cann_sample():
    """The CANN sample's inputs (grad = 1, x = 1..6, beta = 1.1, fp32) against the oracle."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "swishgrad_cann_sample.json")) as f:
        case = json.load(f)
    grad = torch.tensor(case["grad"], dtype=torch.float32, device="cuda").reshape(case["shape"])
    x = torch.tensor(case["x"], dtype=torch.float32, device="cuda").reshape(case["shape"])
    out = _swg().swish_grad(grad, x, case["beta"])
    ref = oracle.swish_grad(np.array(case["grad"], float), np.array(case["x"], float), case["beta"])
    got = to_f64(out).ravel()
    assert np.max(np.abs(got - ref) / np.abs(ref)) < 1e-5
