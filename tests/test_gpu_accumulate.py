"""Accumulate mode of the whole backward (SWG_ACCUMULATE) through the C ABI.

The pages' b and w kernels add db and dw into outputs the caller zeroed
("Kernel signatures" of the SwiGLU backward walk-through), so that several
micro-batches can be summed. With the flag, db_g, db_fc, dw_g, dw_fc become
bf16(old + this call's sum) with one rounding; dx, dg, dfc are overwritten as
without it. Checked here, for both chains, on shapes that take the direct
bf16 epilogue (one M split) and the split-M reduction, and one that runs the
fused chain's side stream (the w stage's reduction beside the x stage's wave):
* db, dw against old + the oracle's sums (dw from the oracle's w stage fed the
  chain's own bf16 dg, dfc), within the output contract;
* dx, dg, dfc bit-identical to a run without the flag;
* accumulating onto zeros bit-identical to a run without the flag;
* M = 0 leaves the four outputs unchanged.
"""

import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, SwigluShape, swiglu_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

SUMMED = ("db_g", "db_fc", "dw_g", "dw_fc")
# M = 100000 at the pages' K, N takes the fused chain's side split: the x stage's last tiles and the
# w stage's split reduction run on the library's side stream
SHAPES = [SWIGLU_CONFIGS["tiny"][0], SWIGLU_CONFIGS["tail"][4],
          SwigluShape("odd_M2_K520_N264", 2, 520, 264, 9, "tail"),
          SwigluShape("split_M100000", 100000, 512, 1024, 13, "pages")]


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _old_outputs(shape, like, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    old = {}
    for k in SUMMED:
        scale = float(like[k].float().abs().max()) or 1.0
        old[k] = (torch.randn(like[k].shape, generator=gen, device="cuda") * scale).to(torch.bfloat16)
    return old


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_accumulate_adds_into_the_outputs(shape, fused):
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    plain = swg.swiglu_bwd(**inp, fused=fused, return_dg=True)
    old = _old_outputs(shape, plain, seed=shape.seed + 17)
    out = {k: v.clone() for k, v in old.items()}
    res = swg.swiglu_bwd(**inp, fused=fused, return_dg=True, out=out, accumulate=True)
    zeros = {k: torch.zeros_like(v) for k, v in old.items()}
    from_zero = swg.swiglu_bwd(**inp, fused=fused, return_dg=True, out=zeros, accumulate=True)
    swg.swg_check()

    for k in ("dg", "dfc", "dx"):
        assert torch.equal(res[k], plain[k]), f"{k} changed under accumulate"
    for k in SUMMED:
        assert torch.equal(from_zero[k], plain[k]), f"{k}: accumulating onto zeros differs from a plain run"

    h = {k: to_f64(v) for k, v in inp.items()}
    _, _, rdbg, rdbfc = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], to_f64(res["dg"]), to_f64(res["dfc"]))
    ref = dict(db_g=rdbg, db_fc=rdbfc, dw_g=rdwg, dw_fc=rdwfc)
    reps = [compare(k, res[k], to_f64(old[k]) + ref[k].reshape(old[k].shape)) for k in SUMMED]
    assert_all(reps)


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
def test_accumulate_with_no_rows_changes_nothing(fused):
    swg = _swg()
    shape = SWIGLU_CONFIGS["tiny"][0]
    inp = swiglu_inputs(shape, device="cuda")
    inp0 = {k: (v[:0] if k in ("x", "dy", "g", "fc") else v) for k, v in inp.items()}
    plain = swg.swiglu_bwd(**inp, fused=fused, return_dg=False)
    old = _old_outputs(shape, plain, seed=5)
    out = {k: v.clone() for k, v in old.items()}
    res = swg.swiglu_bwd(**inp0, fused=fused, return_dg=False, out=out, accumulate=True)
    swg.swg_check()
    for k in SUMMED:
        assert torch.equal(res[k], old[k]), f"{k} changed by an accumulate call over zero rows"
