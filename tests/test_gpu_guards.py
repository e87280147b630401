"""Guard bands around every output and workspace (GPU).

Each case runs an entry point on a tail or odd shape with its outputs (and
its workspace, sized exactly by the workspace query) placed inside guard bands
(tests/_guard.py), then checks that no byte before or after any buffer
changed and that the results still meet the oracle contract. The shapes are
the ones where an out-of-bounds store would come from: masked row and column
tails of the TMA-store epilogues, the fused w kernel's strided dw stores, the
split-M and column-sum reductions, the GroupNorm kernels' misaligned and
streamed paths, SwishGrad's scalar head and tail, and the host path's chunked
copies.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import SwigluShape, group_norm_inputs, swiglu_fwd_biases, swiglu_inputs, swish_inputs

from ._guard import check_all, guarded, workspace
from ._parity import ATOL_ELEM, ATOL_RED, assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

BF = torch.bfloat16
SHAPES = [SwigluShape(f"tail_M{m}", m, 512, 1024, 2, "tail") for m in (1, 127, 1025)] + [
    SwigluShape("odd_M300_K72_N200", 300, 72, 200, 4, "tail"),
    SwigluShape("odd_M129_K8_N8", 129, 8, 8, 5, "tail"),
    SwigluShape("odd_M2_K520_N264", 2, 520, 264, 6, "tail"),
    SwigluShape("odd_M200_K1032_N136", 200, 1032, 136, 7, "tail"),
    SwigluShape("odd_M4099_K1032_N520", 4099, 1032, 520, 8, "tail"),
]


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _np(inp):
    return {k: to_f64(v) for k, v in inp.items()}


def _stage_reports(h, out):
    """dg, dfc, db against the oracle's b stage; dw, dx against its w and x
    stages fed the chain's own bf16 dg, dfc."""
    rdg, rdfc, rdbg, rdbfc = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    gdg, gdfc = to_f64(out["dg"]), to_f64(out["dfc"])
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], gdg, gdfc)
    rdx = oracle.swiglu_bwd_x(gdg, gdfc, h["w_g"], h["w_fc"])
    return [compare("dg", out["dg"], rdg), compare("dfc", out["dfc"], rdfc), compare("db_g", out["db_g"], rdbg),
            compare("db_fc", out["db_fc"], rdbfc), compare("dw_g", out["dw_g"], rdwg),
            compare("dw_fc", out["dw_fc"], rdwfc), compare("dx", out["dx"], rdx)]


def _outs(M, K, N, fill=0xFF):
    shapes = dict(dg=(M, N), dfc=(M, N), dx=(M, K), dw_g=(K, N), dw_fc=(K, N), db_g=(1, N), db_fc=(1, N))
    return {k: guarded(s, BF, fill=fill) for k, s in shapes.items()}


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_whole_backward_guarded(shape, fused):
    swg = _swg()
    M, K, N = shape.M, shape.K, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    g = _outs(M, K, N)
    ws = workspace(swg.swiglu_bwd_workspace_size(M, K, N, swg.SWG_FUSED if fused else swg.SWG_UNFUSED))
    out = swg.swiglu_bwd(**inp, fused=fused, return_dg=True, out={k: v.t for k, v in g.items()},
                         workspace=ws.t)
    swg.swg_check()
    check_all(g)
    ws.check("workspace")
    assert_all(_stage_reports(_np(inp), out))


@pytest.mark.parametrize("shape", [SHAPES[2], SHAPES[3], SHAPES[7]], ids=lambda s: s.name)
def test_stage_calls_guarded(shape):
    swg = _swg()
    M, K, N = shape.M, shape.K, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    g = _outs(M, K, N)
    wb = workspace(swg.swiglu_bwd_b_workspace_size(M, N))
    ww = workspace(swg.swiglu_bwd_w_workspace_size(M, K, N))
    swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"], g["dg"].t, g["dfc"].t, g["db_g"].t, g["db_fc"].t,
                     workspace=wb.t)
    swg.swiglu_bwd_w(inp["x"], g["dg"].t, g["dfc"].t, g["dw_g"].t, g["dw_fc"].t, workspace=ww.t)
    swg.swiglu_bwd_x(g["dg"].t, g["dfc"].t, inp["w_g"], inp["w_fc"], g["dx"].t)
    swg.swg_check()
    check_all(g)
    wb.check("b workspace")
    ww.check("w workspace")
    assert_all(_stage_reports(_np(inp), {k: v.t for k, v in g.items()}))


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2], SHAPES[4], SHAPES[7]], ids=lambda s: s.name)
def test_fused_stage_calls_guarded(shape):
    swg = _swg()
    M, K, N = shape.M, shape.K, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    g = _outs(M, K, N)
    wf = workspace(swg.swiglu_bwd_w_fused_workspace_size(M, K, N))
    swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"], dx=g["dx"].t, dg=g["dg"].t,
                           dfc=g["dfc"].t)
    swg.swiglu_bwd_w_fused(inp["x"], inp["dy"], inp["g"], inp["fc"], g["dw_g"].t, g["dw_fc"].t, g["db_g"].t,
                           g["db_fc"].t, workspace=wf.t)
    swg.swg_check()
    check_all(g)
    wf.check("fused w workspace")
    assert_all(_stage_reports(_np(inp), {k: v.t for k, v in g.items()}))


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[6]], ids=lambda s: s.name)
def test_accumulate_guarded(shape, fused):
    """Accumulate mode reads and writes dw, db in place: the same guards."""
    swg = _swg()
    M, K, N = shape.M, shape.K, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    g = _outs(M, K, N, fill=0)  # accumulating into zeros gives the overwrite result
    ws = workspace(swg.swiglu_bwd_workspace_size(M, K, N, (swg.SWG_FUSED if fused else 0) | swg.SWG_ACCUMULATE))
    out = swg.swiglu_bwd(**inp, fused=fused, return_dg=True, out={k: v.t for k, v in g.items()},
                         workspace=ws.t, accumulate=True)
    swg.swg_check()
    check_all(g)
    ws.check("workspace")
    assert_all(_stage_reports(_np(inp), out))


@pytest.mark.parametrize("shape", SHAPES[3:], ids=lambda s: s.name)
def test_forward_guarded(shape):
    swg = _swg()
    M, K, N = shape.M, shape.K, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    b_g, b_fc = swiglu_fwd_biases(shape, device="cuda")
    g = {k: guarded((M, N), BF) for k in ("g", "fc", "y")}
    out = swg.swiglu_fwd(inp["x"], inp["w_g"], inp["w_fc"], b_g, b_fc, out={k: v.t for k, v in g.items()})
    swg.swg_check()
    check_all(g)
    ref = oracle.swiglu_fwd(to_f64(inp["x"]), to_f64(inp["w_g"]), to_f64(inp["w_fc"]), to_f64(b_g), to_f64(b_fc))
    assert_all([compare(k, out[k], r) for k, r in zip(("g", "fc", "y"), ref)])


DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


@pytest.mark.parametrize("dtype", list(DT), ids=lambda d: DT[d])
@pytest.mark.parametrize("n,offset", [(1, 0), (7, 3), (4100, 1), (1000003, 5), ((1 << 20) + 7, 0)])
def test_swish_and_act_grad_guarded(n, offset, dtype):
    swg = _swg()
    grad, x = swish_inputs(n, dtype, device="cuda", seed=7)
    g = guarded((n,), dtype, offset_elems=offset)
    swg.swish_grad(grad, x, 1.702, grad_x=g.t)
    torch.cuda.synchronize()
    g.check("swish grad_x")
    reps = [compare("grad_x", g.t, oracle.swish_grad(to_f64(grad), to_f64(x), 1.702), dtype=DT[dtype])]
    for act in ("gelu", "hardswish"):
        a = guarded((n,), dtype, offset_elems=offset)
        swg.act_grad(grad, x, act, grad_x=a.t)
        torch.cuda.synchronize()
        a.check(f"{act} grad_x")
        reps.append(compare("grad_x", a.t, oracle.act_grad(to_f64(grad), to_f64(x), act), dtype=DT[dtype]))
    assert_all(reps)


@pytest.mark.parametrize("dtype", list(DT), ids=lambda d: DT[d])
@pytest.mark.parametrize("shape,offset", [((3, 6, 49, 3), 0), ((5, 12, 33, 4), 1), ((2, 64, 49, 32), 0),
                                          ((1, 4, 200000, 2), 0), ((3, 9, 17, 3), 3), ((64, 32, 64, 32), 0)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else str(v))
def test_group_norm_guarded(shape, offset, dtype):
    swg = _swg()
    N, C, HxW, G = shape
    dy, x, gam = group_norm_inputs(N, C, HxW, G, dtype, device="cuda", seed=9)
    gdx = guarded((N, C, HxW), dtype, offset_elems=offset)
    gdg, gdb = guarded((C,), dtype), guarded((C,), dtype)
    ws = workspace(swg.group_norm_bwd_workspace_size(N, C, HxW, G))
    swg.group_norm_bwd(dy, x, G, gamma=gam, eps=1e-5, dx=gdx.t, dgamma=gdg.t, dbeta=gdb.t, workspace=ws.t)
    swg.swg_check()
    check_all(dict(dx=gdx, dgamma=gdg, dbeta=gdb, workspace=ws))
    rdx, rdg, rdb = oracle.group_norm_bwd(to_f64(dy), to_f64(x), to_f64(gam), G, 1e-5)
    assert_all([compare("gn_dx", gdx.t, rdx, dtype=DT[dtype], atol=ATOL_ELEM),
                compare("dgamma", gdg.t, rdg, dtype=DT[dtype], atol=ATOL_RED),
                compare("dbeta", gdb.t, rdb, dtype=DT[dtype], atol=ATOL_RED)])


def test_noalloc_guarded():
    swg = _swg()
    shape = SHAPES[7]
    M, N = shape.M, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    g = {k: guarded(s, BF) for k, s in dict(dg=(M, N), dfc=(M, N), db_g=(1, N), db_fc=(1, N)).items()}
    swg.swiglu_bwd_b_noalloc(inp["dy"], inp["g"], inp["fc"], *(g[k].t for k in ("dg", "dfc", "db_g", "db_fc")))
    swg.swg_check()
    check_all(g)
    h = _np(inp)
    ref = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    assert_all([compare(k, g[k].t, r) for k, r in zip(("dg", "dfc", "db_g", "db_fc"), ref)])


def test_host_path_guarded():
    """swiglu_bwd_host copies results into caller host buffers chunk by chunk."""
    swg = _swg()
    shape = SwigluShape("host_M70001", 70001, 512, 1024, 0, "pages")
    M, K, N = shape.M, shape.K, shape.N
    inp = swiglu_inputs(shape, device="cuda")
    host = {k: v.cpu().pin_memory() for k, v in inp.items()}
    shapes = dict(dx=(M, K), dw_g=(K, N), dw_fc=(K, N), db_g=(1, N), db_fc=(1, N))
    g = {k: guarded(s, BF, device="cpu") for k, s in shapes.items()}
    ws = workspace(swg.swiglu_bwd_host_workspace_size(M, K, N))
    swg.swiglu_bwd_host(**host, out={k: v.t for k, v in g.items()}, workspace=ws.t)
    torch.cuda.synchronize()
    swg.swg_check()
    check_all(g)
    ws.check("host-path workspace")
    dev = swg.swiglu_bwd(**inp, fused=True, return_dg=False)
    torch.cuda.synchronize()
    assert torch.equal(g["dx"].t, dev["dx"].cpu())
    for k in ("dw_g", "dw_fc", "db_g", "db_fc"):
        a, b = to_f64(g[k].t), to_f64(dev[k])
        assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-6), k
