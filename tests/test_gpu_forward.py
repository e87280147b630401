"""SwiGLU forward (g = x W_g + b_g, fc = x W_fc + b_fc, y = SiLU(g) fc) through
the C ABI vs the fp64 oracle (GPU).

g, fc and y are judged like the backward's GEMM outputs: element-wise
|gpu - ref| <= 1e-3 + 2^-7 |ref| with ref the oracle's fp64 value rounded once
to bf16, plus the scale-aware checks (max error <= 2^-6 max|ref|, relative
L2 <= 2^-8). Large shapes compare sampled rows (the oracle's row of a product
needs only that row of x).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, SwigluShape, swiglu_fwd_biases, swiglu_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

ODD = [SwigluShape("odd_M300_K72_N200", 300, 72, 200, 4, "tail"),
       SwigluShape("odd_M129_K8_N8", 129, 8, 8, 5, "tail"),
       SwigluShape("odd_M2_K520_N264", 2, 520, 264, 6, "tail"),
       SwigluShape("odd_M200_K1032_N136", 200, 1032, 136, 7, "tail")]


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _run(shape, bias, rows=None):
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    b_g, b_fc = swiglu_fwd_biases(shape, device="cuda") if bias else (None, None)
    out = swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], b_g, b_fc)
    swg.swg_check()
    x = inp["x"] if rows is None else inp["x"][torch.as_tensor(rows, device="cuda")]
    rb = [None if b is None else to_f64(b) for b in (b_g, b_fc)]
    g, fc, y = oracle.swiglu_fwd(to_f64(x), to_f64(inp["w_g"]), to_f64(inp["w_fc"]), rb[0], rb[1])
    sel = (lambda t: t) if rows is None else (lambda t: t[torch.as_tensor(rows, device="cuda")])
    return [compare("g", sel(out["g"]), g), compare("fc", sel(out["fc"]), fc), compare("y", sel(out["y"]), y)]


@pytest.mark.parametrize("bias", [True, False], ids=["bias", "no_bias"])
@pytest.mark.parametrize("shape", SWIGLU_CONFIGS["tiny"] + SWIGLU_CONFIGS["tail"][:4] + ODD,
                         ids=lambda s: s.name)
def test_forward(shape, bias):
    assert_all(_run(shape, bias))


@pytest.mark.parametrize("shape", SWIGLU_CONFIGS["pages"] + SWIGLU_CONFIGS["llm"] + SWIGLU_CONFIGS["tail"][4:],
                         ids=lambda s: s.name)
def test_forward_full_size_sampled_rows(shape):
    rng = np.random.default_rng(shape.seed + 202)
    rows = np.unique(np.concatenate([rng.choice(shape.M, size=min(512, shape.M), replace=False),
                                     [0, shape.M - 1]]))
    assert_all(_run(shape, True, rows=rows))


def test_forward_is_deterministic_and_feeds_the_backward():
    swg = _swg()
    shape = SWIGLU_CONFIGS["tail"][3]
    inp = swiglu_inputs(shape, device="cuda")
    b_g, b_fc = swiglu_fwd_biases(shape, device="cuda")
    a = swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], b_g, b_fc)
    b = swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], b_g, b_fc)
    swg.swg_check()
    for k in ("g", "fc", "y"):
        assert torch.equal(a[k], b[k])
    # the forward's g, fc are valid inputs of the backward (same layout and dtype)
    out = swg.swiglu_bwd(inp["x"], inp["w_g"], inp["w_fc"], inp["dy"], a["g"], a["fc"], fused=True)
    swg.swg_check()
    h = {k: to_f64(v) for k, v in dict(dy=inp["dy"], g=a["g"], fc=a["fc"]).items()}
    rdg, rdfc, _, _ = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    assert_all([compare("dg", out["dg"], rdg), compare("dfc", out["dfc"], rdfc)])


@pytest.mark.parametrize("shape", [SwigluShape("zero_M", 0, 64, 128, 0, "pages")], ids=lambda s: s.name)
def test_forward_empty(shape):
    swg = _swg()
    x = torch.empty((0, shape.K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((shape.K, shape.N), dtype=torch.bfloat16, device="cuda")
    out = swg.swiglu_fwd(x, w, w)
    swg.swg_check()
    assert out["y"].shape == (0, shape.N)
