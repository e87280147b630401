"""Sibling activation gradients (SiLU, GELU, HardSwish) through the C ABI vs
the fp64 oracle (GPU).

grad_x is judged like SwishGrad's output: |gpu - ref| <= 1e-4 + 2^-7 |ref|
with ref the oracle's fp64 value rounded once to the I/O dtype, plus the
scale-aware checks. Inputs: the SwishGrad recipe (x ~ 4 N(0,1), which covers
GELU's tails and both HardSwish kinks; grad ~ N(0,1)).
"""

import pytest
import torch

import oracle
from synth import SWISH_CONFIG, swish_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
ACTS = ("silu", "gelu", "hardswish")


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _check(act, grad, x, out):
    ref = oracle.act_grad(to_f64(grad), to_f64(x), act)
    return compare("grad_x", out, ref, dtype=DT[grad.dtype])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
@pytest.mark.parametrize("n", SWISH_CONFIG["n"])
@pytest.mark.parametrize("act", ACTS)
def test_act_grad_full_size(act, n, dtype):
    grad, x = swish_inputs(n, dtype, device="cuda", seed=SWISH_CONFIG["seed"])
    out = _swg().act_grad(grad, x, act)
    torch.cuda.synchronize()
    assert_all([_check(act, grad, x, out)])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
@pytest.mark.parametrize("n", [1, 7, 9, 1000003])
@pytest.mark.parametrize("act", ACTS)
def test_act_grad_small_and_ragged(act, n, dtype):
    grad, x = swish_inputs(n, dtype, device="cuda", seed=8)
    out = _swg().act_grad(grad, x, act)
    torch.cuda.synchronize()
    assert_all([_check(act, grad, x, out)])


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
def test_act_grad_special_values(dtype):
    swg = _swg()
    x = torch.tensor([-40.0, -4.0, -3.0, 0.0, 3.0, 4.0, 40.0], dtype=dtype, device="cuda")
    grad = torch.full_like(x, 2.0)
    h = swg.act_grad(grad, x, "hardswish").float().cpu().tolist()
    assert h == [0.0, 0.0, 0.0, 1.0, 2.0, 2.0, 2.0]
    g = swg.act_grad(grad, x, "gelu").float().cpu()
    assert g[3].item() == 1.0 and g[6].item() == 2.0 and g[0].item() == 0.0


@pytest.mark.parametrize("dtype", SWISH_CONFIG["dtypes"], ids=lambda d: DT[d])
def test_silu_is_swish_grad_with_beta_one_and_in_place(dtype):
    swg = _swg()
    grad, x = swish_inputs(100003, dtype, device="cuda", seed=9)
    a = swg.act_grad(grad, x, "silu")
    b = swg.swish_grad(grad, x, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    g2 = grad.clone()
    swg.act_grad(g2, x, "gelu", grad_x=g2)  # grad_x aliasing grad exactly
    torch.cuda.synchronize()
    assert_all([_check("gelu", grad, x, g2)])


def test_act_grad_rejects_unknown_activation():
    swg = _swg()
    t = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        swg.act_grad(t, t, "relu")


def test_bindings_refuse_outputs_that_would_be_overrun():
    swg = _swg()
    g, x = swish_inputs(1000, torch.bfloat16, device="cuda", seed=3)
    for bad in (torch.empty(999, dtype=torch.bfloat16, device="cuda"),         # short
                torch.empty(1000, dtype=torch.float32, device="cuda"),         # wrong dtype
                torch.empty(2000, dtype=torch.bfloat16, device="cuda")[::2],   # strided
                torch.empty(1000, dtype=torch.bfloat16)):                       # host memory
        with pytest.raises(ValueError):
            swg.act_grad(g, x, "gelu", grad_x=bad)
        with pytest.raises(ValueError):
            swg.swish_grad(g, x, 1.0, grad_x=bad)
    dy, xx, gam = (t.cuda() for t in __import__("synth").group_norm_inputs(2, 8, 12, 4, torch.float16, seed=1))
    with pytest.raises(ValueError):
        swg.group_norm_bwd(dy, xx, 4, gamma=gam, dgamma=torch.empty(7, dtype=torch.float16, device="cuda"))
    from synth import SWIGLU_CONFIGS, swiglu_inputs
    inp = swiglu_inputs(SWIGLU_CONFIGS["tiny"][0], device="cuda")
    M, K = inp["x"].shape
    with pytest.raises(ValueError):
        swg.swiglu_bwd(**inp, out={"dx": torch.empty(M - 1, K, dtype=torch.bfloat16, device="cuda")})
