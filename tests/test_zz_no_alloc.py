"""swiglu_bwd_b_noalloc: the b stage for callers that cannot allocate.

Such callers (a framework whose memory pool owns all of device memory, a loop
that cannot afford cudaMalloc's implicit synchronisation) get an entry point
whose column partials live in a fixed array inside the library instead of a
caller workspace. This file is collected last so that a run stopping at the
first failure has already run every other test; it also passes on its own.
"""

import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, swiglu_inputs

from ._parity import assert_all, compare, to_f64


def test_noalloc_rejects_shapes_beyond_the_array():
    """N > 524288 needs more partials than the array holds: refused up front."""
    from swiglu_ffn_backward_gb300 import _binding as b
    base = 0x7f0000000000
    N = 1 << 20
    M = 8
    p = [base + i * (1 << 28) for i in range(7)]
    assert b.lib.swiglu_bwd_b_noalloc(*p, M, N, None) == b.SWG_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row, on different inputs and sizes, each against the fp64 oracle's b stage and
    bit for bit against swiglu_bwd_b."""
    import swiglu_ffn_backward_gb300 as swg
    for shape in (SWIGLU_CONFIGS["tail"][3], SWIGLU_CONFIGS["tail"][2]):  # M=4097, then M=1025
        inp = swiglu_inputs(shape, device="cuda")
        ref = swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"])
        got = swg.swiglu_bwd_b_noalloc(inp["dy"], inp["g"], inp["fc"])
        swg.swg_check()
        names = ("dg", "dfc", "db_g", "db_fc")
        expect = oracle.swiglu_bwd_b(to_f64(inp["dy"]), to_f64(inp["g"]), to_f64(inp["fc"]))
        assert_all([compare(n, gt, ex) for n, gt, ex in zip(names, got, expect)])
        for gt, rf in zip(got, ref):  # same kernel, same plan: the same bits
            assert torch.equal(gt, rf)


@pytest.mark.gpu
def test_noalloc_at_the_array_limit_and_empty():
    """N = 524288 fills the array exactly (one partial row pair of 8N bytes);
    M = 0 writes zero column sums. Both against swiglu_bwd_b, twice in a row."""
    import swiglu_ffn_backward_gb300 as swg
    from synth import SwigluShape
    shape = SwigluShape("noalloc_limit", 8, 8, 524288, 3, "tail")
    inp = swiglu_inputs(shape, device="cuda")
    for _ in range(2):
        ref = swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"])
        got = swg.swiglu_bwd_b_noalloc(inp["dy"], inp["g"], inp["fc"])
        swg.swg_check()
        for gt, rf in zip(got, ref):
            assert torch.equal(gt, rf)
    z = torch.empty((0, 1024), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        dg, dfc, db_g, db_fc = swg.swiglu_bwd_b_noalloc(z, z, z)
        swg.swg_check()
        assert dg.numel() == 0 and dfc.numel() == 0
        assert torch.count_nonzero(db_g).item() == 0 and torch.count_nonzero(db_fc).item() == 0
