"""The bf16 values the GPU picks for dg and dfc are valid roundings (GPU).

dg and dfc are computed in fp32 and rounded once to bf16; the oracle rounds
the exact (fp64) value. The two differ only where the exact value lies so
close to the midpoint between two neighbouring bf16 values that the fp32
arithmetic error decides the side. This test checks exactly that, element by
element: every GPU value either equals the oracle's round-to-nearest-even of
the exact value, or is the other neighbour of the exact value and the exact
value lies within 2^-16 of the computation's scale from the midpoint (about
a hundred fp32 roundings; a bf16 spacing is 2^-8 to 2^-7 of a value). The
scale is the magnitude of the terms: |dy fc| s (1 + |g| (1 - s)) for dg,
whose bracket cancels near g = -1.28, and |dy g s| for dfc (s = sigma(g)). Both
choices are correct roundings of a value that fp32 arithmetic cannot place
on one side, which is why the w and x stages are judged on the chain's own
dg, dfc (the rest of the chain is then checked against the oracle fed those
valid choices).
"""

import numpy as np
import pytest
import torch

import oracle
from oracle.numerics import bf16_bits_to_f64, f64_to_bf16_bits
from synth import SWIGLU_CONFIGS, swiglu_inputs

from ._parity import to_f64

pytestmark = pytest.mark.gpu

TIE_TOL = 2.0 ** -16


def _neighbour_away(r_bits, exact, r):
    """The bf16 neighbour of r (bit patterns of finite values) on the side of exact."""
    b = r_bits.astype(np.int32)
    toward_larger = exact > r
    positive = (b & 0x8000) == 0  # larger values: larger bit patterns for positive, smaller for negative
    nb = np.where(positive, np.where(toward_larger, b + 1, b - 1), np.where(toward_larger, b - 1, b + 1))
    nb = np.where((r == 0) & toward_larger, 0x0001, nb)
    nb = np.where((r == 0) & ~toward_larger, 0x8001, nb)
    return bf16_bits_to_f64(nb.astype(np.uint16))


def _check_choices(gpu, exact, scale):
    r_bits = f64_to_bf16_bits(exact)
    r = bf16_bits_to_f64(r_bits)
    g = to_f64(gpu).reshape(exact.shape)
    diff = g != r
    n_diff = int(np.count_nonzero(diff))
    if n_diff:
        e, rr, gg, rb, sc = exact[diff], r[diff], g[diff], r_bits[diff], scale[diff]
        other = _neighbour_away(rb, e, rr)
        assert np.all(gg == other), "a GPU value is neither rounding neighbour of the exact value"
        mid = 0.5 * (rr + other)
        assert np.all(np.abs(e - mid) <= TIE_TOL * sc), \
            f"a GPU rounding differs away from a tie: max {np.max(np.abs(e - mid) / sc):.3g} of the scale"
    return n_diff / exact.size


@pytest.mark.parametrize("shape", [SWIGLU_CONFIGS["tiny"][0], SWIGLU_CONFIGS["tail"][3], SWIGLU_CONFIGS["tail"][4]],
                         ids=lambda s: s.name)
@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
def test_dg_dfc_rounding_choices_are_valid(shape, fused):
    import swiglu_ffn_backward_gb300 as swg
    inp = swiglu_inputs(shape, device="cuda")
    out = swg.swiglu_bwd(**inp, fused=fused, return_dg=True)
    torch.cuda.synchronize()
    swg.swg_check()
    dy, g, fc = to_f64(inp["dy"]), to_f64(inp["g"]), to_f64(inp["fc"])
    dg, dfc, _, _ = oracle.swiglu_bwd_b(dy, g, fc)
    s = oracle.sigmoid(g)
    f_dg = _check_choices(out["dg"], dg, np.abs(dy * fc) * s * (1.0 + np.abs(g) * (1.0 - s)))
    f_dfc = _check_choices(out["dfc"], dfc, np.abs(dfc))
    # near-ties are rare: well under 1% of the elements
    assert f_dg < 0.01 and f_dfc < 0.01, (f_dg, f_dfc)
