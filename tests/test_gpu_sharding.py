"""Sharding the backward along M, checked on one GPU.

The path is data parallel over rows (tokens): dg, dfc and dx of a row depend
on that row only, while db and dw are sums over all rows. A run split into
M-slices must therefore reproduce the row-local outputs of the unsharded run
exactly. For db and dw, each slice returns its own sum rounded to bf16; adding
them (what an all-reduce of the outputs over ranks would form) differs from
the unsharded result by the roundings alone: each bf16 rounding moves a value
by at most 2^-8 of its magnitude, so the sum of the slices must lie within
1e-3 + 2^-8 * (sum of |slice values| + |unsharded value|) of the unsharded
value, element by element (where slices cancel, this is looser than the
output contract, which is why a multi-GPU version would reduce the fp32
partials before rounding). The relative L2 error must also stay within 2^-8.
Both the unfused and the fused chain are checked, with cuts on a 128-row tile
boundary and inside tiles.
"""

import pytest
import torch

from synth import SWIGLU_CONFIGS, swiglu_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

ROW_LOCAL = ("dg", "dfc", "dx")
SUMMED = ("db_g", "db_fc", "dw_g", "dw_fc")


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _run(swg, inp, fused):
    out = swg.swiglu_bwd(**inp, fused=fused, return_dg=True)
    swg.swg_check()
    return out


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
@pytest.mark.parametrize("cuts", [(2048,), (1000, 3001)], ids=["tile_aligned", "inside_tiles"])
def test_m_shards_reproduce_the_unsharded_backward(cuts, fused):
    swg = _swg()
    shape = SWIGLU_CONFIGS["tail"][3]  # M=4097, K=512, N=1024, saturating g
    inp = swiglu_inputs(shape, device="cuda")
    M = shape.M
    full = _run(swg, inp, fused)
    bounds = [0, *cuts, M]
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        sl = dict(inp)
        for k in ("x", "dy", "g", "fc"):
            sl[k] = inp[k][a:b]
        parts.append(_run(swg, sl, fused))
    torch.cuda.synchronize()

    aligned = all(c % 128 == 0 for c in cuts)
    reps = []
    for k in ROW_LOCAL:
        cat = torch.cat([p[k] for p in parts])
        if k != "dx" or aligned:
            # element-wise math, or the same tile positions: bit-identical
            assert torch.equal(cat, full[k]), f"{k}: sharded rows differ from the unsharded run"
        else:
            reps.append(compare(k, cat, to_f64(full[k])))
    for k in SUMMED:
        shards = [p[k].double() for p in parts]
        ref = full[k].double()
        total = sum(shards)  # the reduction over shards
        err = (total - ref).abs()
        bound = 1e-3 + 2.0 ** -8 * (sum(t.abs() for t in shards) + ref.abs())
        n_bad = int((~(err <= bound)).sum())
        assert n_bad == 0, f"{k}: {n_bad} elements outside the rounding bound (max err {float(err.max()):.3g})"
        rel_l2 = float(torch.linalg.norm(total - ref) / torch.linalg.norm(ref))
        assert rel_l2 <= 2.0 ** -8, f"{k}: relative L2 error {rel_l2:.3g}"
    assert_all(reps)
