"""The timeout path of the tcgen05 kernels' bounded pipeline waits.

Every mbarrier wait in the GEMM pipelines gives up after a cycle limit, sets
the library's status word and lets the kernel stop, drain what it issued, free
its tensor memory and return, so that a lost arrival becomes SWG_ERR_TIMEOUT
from swg_check() instead of a hung GPU. These tests make that happen on
purpose, on the host's terms: swg_inject_stall arms the next launch of one
kernel so that its operand producer stops issuing copies before a given ring
entry (nothing is left in flight) and its waits give up after about half a
millisecond. The consumer's wait on the missing entry runs out; the test
checks the status, then runs the same call again and checks it against the
oracle, which shows the GPU and the library still work normally.
"""

import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, SwigluShape, swiglu_inputs

from ._parity import assert_all, compare, to_f64

LIMIT = 1 << 20  # cycles, about half a millisecond


def test_injection_arguments_are_checked():
    from swiglu_ffn_backward_gb300 import _binding as b
    assert b.lib.swg_inject_stall(7, 1, LIMIT) == b.SWG_ERR_PARAM_INVALID
    assert b.lib.swg_inject_stall(5, 1, LIMIT) == b.SWG_ERR_PARAM_INVALID
    assert b.lib.swg_inject_stall(b.SWG_INJECT_X_GEMM, -1, LIMIT) == b.SWG_ERR_PARAM_INVALID
    assert b.lib.swg_inject_stall(b.SWG_INJECT_X_GEMM, 1, 100) == b.SWG_ERR_PARAM_INVALID
    # arming and disarming touches host state only
    assert b.lib.swg_inject_stall(b.SWG_INJECT_FUSED_X, 3, LIMIT) == b.SWG_OK
    assert b.lib.swg_inject_stall(b.SWG_INJECT_FUSED_W, 0, LIMIT) == b.SWG_OK
    assert b.lib.swg_inject_stall(b.SWG_INJECT_FWD, 2, LIMIT) == b.SWG_OK
    assert b.lib.swg_inject_stall(0, 0, 0) == b.SWG_OK


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _expect_timeout(swg):
    with pytest.raises(swg.SwgError) as e:
        swg.swg_check()
    assert e.value.status == 6  # SWG_ERR_TIMEOUT
    swg.swg_check()  # the status word was cleared


@pytest.mark.gpu
@pytest.mark.parametrize("entry", [0, 1, 3])
def test_x_gemm_wait_runs_out(entry):
    swg = _swg()
    inp = swiglu_inputs(SWIGLU_CONFIGS["tiny"][0], device="cuda")  # 4 ring entries per tile
    dg, dfc, _, _ = swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"])
    swg.swg_check()
    swg.swg_inject_stall(swg.SWG_INJECT_X_GEMM, entry, LIMIT)
    swg.swiglu_bwd_x(dg, dfc, inp["w_g"], inp["w_fc"])
    _expect_timeout(swg)
    dx = swg.swiglu_bwd_x(dg, dfc, inp["w_g"], inp["w_fc"])
    swg.swg_check()
    ref = oracle.swiglu_bwd_x(to_f64(dg), to_f64(dfc), to_f64(inp["w_g"]), to_f64(inp["w_fc"]))
    assert_all([compare("dx", dx, ref)])


@pytest.mark.gpu
@pytest.mark.parametrize("entry", [0, 1, 3])
def test_fused_x_wait_runs_out(entry):
    swg = _swg()
    shape = SWIGLU_CONFIGS["tiny"][0]  # one tile per CTA: two stages, four ring entries in all
    inp = swiglu_inputs(shape, device="cuda")
    swg.swg_inject_stall(swg.SWG_INJECT_FUSED_X, entry, LIMIT)
    swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"])
    _expect_timeout(swg)
    out = swg.swiglu_bwd(**inp, fused=True)
    swg.swg_check()
    h = {k: to_f64(v) for k, v in inp.items()}
    rdx = oracle.swiglu_bwd_x(to_f64(out["dg"]), to_f64(out["dfc"]), h["w_g"], h["w_fc"])
    assert_all([compare("dx", out["dx"], rdx)])
    torch.cuda.synchronize()


@pytest.mark.gpu
@pytest.mark.parametrize("entry", [0, 1, 3])
def test_fused_w_wait_runs_out(entry):
    """The fused w kernel runs on CTA pairs (M=2048 K=64 N=128: four M-splits of one pair of
    64-column bands, eight stages per CTA, four stage slots). Both CTAs' producers stop before the
    entry; the leader's MMA wait runs out; the transform warps' waits for the slots of the stages
    four on run out too, and those warps arrive only on slots whose previous use was released; both
    CTAs meet at the final cluster barrier. A normal call afterwards passes."""
    swg = _swg()
    shape = SwigluShape("fw_stall_M2048", 2048, 64, 128, 9, "tail")
    inp = swiglu_inputs(shape, device="cuda")
    swg.swg_inject_stall(swg.SWG_INJECT_FUSED_W, entry, LIMIT)
    swg.swiglu_bwd_w_fused(inp["x"], inp["dy"], inp["g"], inp["fc"])
    _expect_timeout(swg)
    out = swg.swiglu_bwd(**inp, fused=True)
    swg.swg_check()
    h = {k: to_f64(v) for k, v in inp.items()}
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], to_f64(out["dg"]), to_f64(out["dfc"]))
    assert_all([compare("dw_g", out["dw_g"], rdwg), compare("dw_fc", out["dw_fc"], rdwfc)])
    torch.cuda.synchronize()


@pytest.mark.gpu
@pytest.mark.parametrize("entry", [0, 1, 7])
def test_forward_wait_runs_out(entry):
    """The forward runs on CTA pairs (M=1024 K=512 N=256: eight pair tiles, one per pair, eight
    K blocks each, six stage slots). Both CTAs' producers stop before the entry; the leader's MMA
    wait runs out, then both CTAs' epilogue waits; both CTAs meet at the final cluster barriers. A
    normal call afterwards matches the oracle."""
    from synth import swiglu_fwd_biases
    swg = _swg()
    shape = SwigluShape("fwd_stall_M1024", 1024, 512, 256, 21, "tail")
    inp = swiglu_inputs(shape, device="cuda")
    b_g, b_fc = swiglu_fwd_biases(shape, device="cuda")
    swg.swg_inject_stall(swg.SWG_INJECT_FWD, entry, LIMIT)
    swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], b_g, b_fc)
    _expect_timeout(swg)
    out = swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], b_g, b_fc)
    swg.swg_check()
    g, fc, y = oracle.swiglu_fwd(to_f64(inp["x"]), to_f64(inp["w_g"]), to_f64(inp["w_fc"]), to_f64(b_g),
                                 to_f64(b_fc))
    assert_all([compare("g", out["g"], g), compare("fc", out["fc"], fc), compare("y", out["y"], y)])
    torch.cuda.synchronize()
