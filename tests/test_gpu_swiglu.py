"""SwiGLU-FFN backward through the C ABI vs the fp64 oracle (GPU).

Inputs are drawn once on the GPU from the seeded recipes in `synth` and copied
to the host for the oracle, so both sides see the same bf16 bits.

How each output is judged:
* dg, dfc, db_g, db_fc: element-wise contract against the oracle's b stage.
* dw_g, dw_fc, dx: element-wise contract against the oracle's w and x stages
  fed the bf16 dg, dfc that the chain itself produced (returned alongside).
  Those dg, dfc pass the contract against the oracle, but where the GPU's fp32
  value and the oracle's fp64 value fall on opposite sides of a bf16 rounding
  boundary they differ by one bf16 ulp, and a GEMM output summing many such
  elements can move by one or two of its own ulps; feeding the oracle the
  chain's dg isolates the GEMM's own error.
* dw_g, dw_fc, dx against the oracle's whole backward (its own bf16 rounding
  of dg, dfc) and against the exact gradient (no rounding of dg, dfc): the
  scale-aware norm checks (max error <= 2^-6 max|ref|, relative L2 <= 2^-8).
"""

import numpy as np
import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, SwigluShape, swiglu_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

FULL_ORACLE_MAX_MN = 5_000_000  # above this, sample rows/columns


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _np(inp):
    return {k: to_f64(v) for k, v in inp.items()}


def _norm_only(rep, suffix):
    rep["ok"] = rep["finite"] and rep["max_err"] <= 2.0 ** -6 * rep["max_ref"] and rep["rel_l2"] <= 2.0 ** -8
    rep["name"] += suffix
    return rep


def _full_case(shape: SwigluShape, fused: bool):
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    out = swg.swiglu_bwd(**inp, fused=fused, return_dg=True)
    swg.swg_check()
    h = _np(inp)
    rdg, rdfc, rdbg, rdbfc = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    reps = [compare("dg", out["dg"], rdg), compare("dfc", out["dfc"], rdfc),
            compare("db_g", out["db_g"], rdbg), compare("db_fc", out["db_fc"], rdbfc)]
    gdg, gdfc = to_f64(out["dg"]), to_f64(out["dfc"])
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], gdg, gdfc)
    rdx = oracle.swiglu_bwd_x(gdg, gdfc, h["w_g"], h["w_fc"])
    reps += [compare("dw_g", out["dw_g"], rdwg), compare("dw_fc", out["dw_fc"], rdwfc),
             compare("dx", out["dx"], rdx)]
    for stage_dtype, suffix in (("bf16", "(oracle chain)"), (None, "(exact)")):
        ref = oracle.swiglu_bwd(h["x"], h["w_g"], h["w_fc"], h["dy"], h["g"], h["fc"], stage_dtype=stage_dtype)
        for k in ("dw_g", "dw_fc", "dx"):
            reps.append(_norm_only(compare(k, out[k], ref[k]), suffix))
    return reps


def _sampled_case(shape: SwigluShape, fused: bool, n_rows=384, n_cols=96):
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    out = swg.swiglu_bwd(**inp, fused=fused, return_dg=True)
    swg.swg_check()
    rng = np.random.default_rng(shape.seed + 101)
    M, N = shape.M, shape.N
    rows = np.unique(np.concatenate([rng.choice(M, size=min(n_rows, M), replace=False), [0, M - 1]]))
    cols = np.unique(np.concatenate([rng.choice(N, size=min(n_cols, N), replace=False), [0, N - 1]]))
    rt = torch.as_tensor(rows, device="cuda")
    ct = torch.as_tensor(cols, device="cuda")
    cpu = {k: v.cpu() for k, v in inp.items()}
    # b stage on the sampled rows and columns
    ref = oracle.swiglu_bwd_sampled(cpu["x"], cpu["w_g"], cpu["w_fc"], cpu["dy"], cpu["g"], cpu["fc"],
                                    rows, cols, stage_dtype="bf16")
    reps = [compare("dg", out["dg"][rt], ref["dg"]), compare("dfc", out["dfc"][rt], ref["dfc"]),
            compare("db_g", out["db_g"][:, ct], ref["db_g"]), compare("db_fc", out["db_fc"][:, ct], ref["db_fc"])]
    # w and x stages fed the chain's own dg, dfc (rows for dx, columns for dw)
    x64 = to_f64(inp["x"])
    rdx = oracle.swiglu_bwd_x(to_f64(out["dg"][rt]), to_f64(out["dfc"][rt]), to_f64(inp["w_g"]),
                              to_f64(inp["w_fc"]))
    rdwg, rdwfc = oracle.swiglu_bwd_w(x64, to_f64(out["dg"][:, ct]), to_f64(out["dfc"][:, ct]))
    reps += [compare("dx", out["dx"][rt], rdx), compare("dw_g", out["dw_g"][:, ct], rdwg),
             compare("dw_fc", out["dw_fc"][:, ct], rdwfc)]
    # the oracle's own chain: norm checks
    reps += [_norm_only(compare("dx", out["dx"][rt], ref["dx"]), "(oracle chain)"),
             _norm_only(compare("dw_g", out["dw_g"][:, ct], ref["dw_g"]), "(oracle chain)"),
             _norm_only(compare("dw_fc", out["dw_fc"][:, ct], ref["dw_fc"]), "(oracle chain)")]
    return reps


def _shapes(names):
    return [s for n in names for s in SWIGLU_CONFIGS[n]]


FUSED = pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])


@FUSED
@pytest.mark.parametrize("shape", _shapes(["tiny", "tail"]), ids=lambda s: s.name)
def test_swiglu_bwd(shape, fused):
    if shape.M * shape.N <= FULL_ORACLE_MAX_MN:
        assert_all(_full_case(shape, fused=fused))
    else:
        assert_all(_sampled_case(shape, fused=fused))


@FUSED
@pytest.mark.parametrize("shape", _shapes(["pages", "llm"]), ids=lambda s: s.name)
def test_swiglu_bwd_full_size(shape, fused):
    assert_all(_sampled_case(shape, fused=fused))


ODD = [SwigluShape("odd_M300_K72_N200", 300, 72, 200, 4, "tail"),
       SwigluShape("odd_M129_K8_N8", 129, 8, 8, 5, "tail"),
       SwigluShape("odd_M2_K520_N264", 2, 520, 264, 6, "tail")]


@FUSED
@pytest.mark.parametrize("shape", ODD + [SwigluShape("odd_M200_K1032_N136", 200, 1032, 136, 7, "tail")],
                         ids=lambda s: s.name)
def test_swiglu_bwd_odd_shapes(shape, fused):
    assert_all(_full_case(shape, fused=fused))


@pytest.mark.parametrize("shape", _shapes(["tiny"]) + [SWIGLU_CONFIGS["tail"][2], ODD[0]], ids=lambda s: s.name)
def test_stage_calls(shape):
    """b, then w and x on the GPU's own bf16 dg, dfc (stage oracles)."""
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    dg, dfc, db_g, db_fc = swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"])
    dw_g, dw_fc = swg.swiglu_bwd_w(inp["x"], dg, dfc)
    dx = swg.swiglu_bwd_x(dg, dfc, inp["w_g"], inp["w_fc"])
    swg.swg_check()
    h = _np(inp)
    rdg, rdfc, rdbg, rdbfc = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    gdg, gdfc = to_f64(dg), to_f64(dfc)
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], gdg, gdfc)
    rdx = oracle.swiglu_bwd_x(gdg, gdfc, h["w_g"], h["w_fc"])
    assert_all([compare("dg", dg, rdg), compare("dfc", dfc, rdfc), compare("db_g", db_g, rdbg),
                compare("db_fc", db_fc, rdbfc), compare("dw_g", dw_g, rdwg), compare("dw_fc", dw_fc, rdwfc),
                compare("dx", dx, rdx)])


@pytest.mark.parametrize("shape", _shapes(["tiny"]) + [SWIGLU_CONFIGS["tail"][2], ODD[0]], ids=lambda s: s.name)
def test_fused_stage_calls(shape):
    """The fused x and w stages called separately; dw, dx against the oracle's
    stages fed the b stage's bf16 dg, dfc, which the fused kernels reproduce."""
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    dx, dg, dfc = swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"], return_dg=True)
    dx2, _, _ = swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"])
    dw_g, dw_fc, db_g, db_fc = swg.swiglu_bwd_w_fused(inp["x"], inp["dy"], inp["g"], inp["fc"])
    swg.swg_check()
    h = _np(inp)
    rdg, rdfc, rdbg, rdbfc = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    gdg, gdfc = to_f64(dg), to_f64(dfc)
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], gdg, gdfc)
    rdx = oracle.swiglu_bwd_x(gdg, gdfc, h["w_g"], h["w_fc"])
    assert_all([compare("dg", dg, rdg), compare("dfc", dfc, rdfc), compare("db_g", db_g, rdbg),
                compare("db_fc", db_fc, rdbfc), compare("dw_g", dw_g, rdwg), compare("dw_fc", dw_fc, rdwfc),
                compare("dx", dx, rdx)])
    # without the optional dg, dfc outputs dx is the same bits
    assert torch.equal(dx, dx2)


@pytest.mark.parametrize("shape", [SWIGLU_CONFIGS["tail"][3], ODD[0]], ids=lambda s: s.name)
def test_fused_operands_match_b_stage_bits(shape):
    """dg, dfc formed on chip by the fused kernel are bit-identical to the b stage's."""
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    dg, dfc, _, _ = swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"])
    _, fdg, fdfc = swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"],
                                          return_dg=True)
    swg.swg_check()
    assert torch.equal(dg, fdg) and torch.equal(dfc, fdfc)


def test_empty_M_writes_zero_sums():
    swg = _swg()
    K, N = 64, 128
    z = lambda *s: torch.empty(s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    out = dict(dx=z(0, K), dw_g=z(K, N).fill_(7), dw_fc=z(K, N).fill_(7), db_g=z(1, N).fill_(7),
               db_fc=z(1, N).fill_(7), dg=z(0, N), dfc=z(0, N))
    for fused in (False, True):
        for k in ("dw_g", "dw_fc", "db_g", "db_fc"):
            out[k].fill_(7)
        swg.swiglu_bwd(z(0, K), z(K, N), z(K, N), z(0, N), z(0, N), z(0, N), out=out, fused=fused)
        torch.cuda.synchronize()
        for k in ("dw_g", "dw_fc", "db_g", "db_fc"):
            assert torch.count_nonzero(out[k]) == 0, (k, fused)


def test_db_equals_sum_of_dg_and_linearity():
    """db_g agrees with the fp64 sum of the GPU's dg (up to dg's bf16 rounding),
    and doubling dy doubles every output exactly."""
    swg = _swg()
    shape = SWIGLU_CONFIGS["tail"][3]  # M=4097
    inp = swiglu_inputs(shape, device="cuda")
    a = swg.swiglu_bwd(**inp)
    inp2 = dict(inp, dy=inp["dy"] * 2)
    b = swg.swiglu_bwd(**inp2)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(b[k].float(), a[k].float() * 2), k
    s = to_f64(a["dg"]).sum(axis=0)
    db = to_f64(a["db_g"]).ravel()
    # each bf16 dg is within 2^-9 relative of the fp32 value that db sums
    slack = 2.0 ** -9 * np.abs(to_f64(a["dg"])).sum(axis=0) + 2.0 ** -8 * np.abs(db) + 1e-6
    assert np.all(np.abs(s - db) <= slack)


@FUSED
def test_deterministic(fused):
    swg = _swg()
    inp = swiglu_inputs(SWIGLU_CONFIGS["tail"][3], device="cuda")
    a = swg.swiglu_bwd(**inp, fused=fused)
    b = swg.swiglu_bwd(**inp, fused=fused)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("shape", [SWIGLU_CONFIGS["tail"][3], SWIGLU_CONFIGS["tail"][4]], ids=lambda s: s.name)
def test_auto_chain_is_the_chosen_chain(shape):
    """fused=None (SWG_AUTO) gives exactly the bits of the chain it selects: unfused at
    M = 4097, fused at M = 65537 (K = 512)."""
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    a = swg.swiglu_bwd(**inp)
    b = swg.swiglu_bwd(**inp, fused=shape.M >= 32768)
    swg.swg_check()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.gpu
def test_w_stage_many_tiles_per_cta():
    """The w GEMM with more dw tiles than CTAs (K = 2048, N = 2560: 2 x 16 x 10 = 320 tiles of 128 x 256
    and no M split at M = 384): each persistent CTA takes two or three tiles through both TMEM
    accumulators, and the column tiles form a group of eight and a short group of two. Against the
    w-stage oracle on the GPU's own dg, dfc, then once more in accumulate mode on top of the result."""
    swg = _swg()
    shape = SwigluShape("w_many_tiles", 384, 2048, 2560, 7, "tail")
    inp = swiglu_inputs(shape, device="cuda")
    dg, dfc, _, _ = swg.swiglu_bwd_b(inp["dy"], inp["g"], inp["fc"])
    dw_g, dw_fc = swg.swiglu_bwd_w(inp["x"], dg, dfc)
    swg.swg_check()
    h = _np(inp)
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], to_f64(dg), to_f64(dfc))
    assert_all([compare("dw_g", dw_g, rdwg), compare("dw_fc", dw_fc, rdwfc)])
    # the same call through swiglu_bwd's accumulate mode adds a second copy of the sums onto dw
    outs = swg.swiglu_bwd(**inp, fused=False)
    base = {k: v.clone() for k, v in outs.items()}
    swg.swiglu_bwd(**inp, fused=False, accumulate=True, out=outs)
    swg.swg_check()
    for k in ("dw_g", "dw_fc"):
        ref = 2.0 * to_f64(base[k])
        assert_all([compare(k, outs[k], ref)])


@pytest.mark.gpu
@pytest.mark.parametrize("N", [1024, 1000])
def test_fused_chain_side_split_matches_stage_calls(N):
    """At M = 100000, K = 512, N = 1024 the fused whole-backward call runs the x stage's last tiles
    beside the w stage (the w stage leaves SMs free and the x stage needs six waves), and the w
    stage's reduction on the side stream beside the x stage's wave: every output must equal the two
    stage calls' bit for bit. N = 1000 leaves a ragged last column band. The outputs start filled
    with a value no result takes, so a tile the split left out would show."""
    swg = _swg()
    shape = SwigluShape(f"split_M100000_N{N}", 100000, 512, N, 11, "pages")
    inp = swiglu_inputs(shape, device="cuda")
    M, K, N = shape.M, shape.K, shape.N
    # FW, its reduction, and the x stage in two launches: the side stream is in use
    assert swg.swiglu_bwd_kernel_count(M, K, N, swg.SWG_FUSED) == 4
    bf = dict(dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), **bf)
    swg.swiglu_bwd_x_fused(inp["dy"], inp["g"], inp["fc"], inp["w_g"], inp["w_fc"], dx)
    dwg, dwfc = torch.empty((K, N), **bf), torch.empty((K, N), **bf)
    dbg, dbfc = torch.empty((1, N), **bf), torch.empty((1, N), **bf)
    ws = torch.empty(max(swg.swiglu_bwd_w_fused_workspace_size(M, K, N), 16), dtype=torch.uint8, device="cuda")
    swg.swiglu_bwd_w_fused(inp["x"], inp["dy"], inp["g"], inp["fc"], dwg, dwfc, dbg, dbfc, workspace=ws)
    out = {"dx": torch.full((M, K), 3.0e38, **bf), "dw_g": torch.full((K, N), 3.0e38, **bf),
           "dw_fc": torch.full((K, N), 3.0e38, **bf), "db_g": torch.full((1, N), 3.0e38, **bf),
           "db_fc": torch.full((1, N), 3.0e38, **bf)}
    swg.swiglu_bwd(**inp, fused=True, return_dg=False, out=out)
    swg.swg_check()
    for name, ref in (("dx", dx), ("dw_g", dwg), ("dw_fc", dwfc), ("db_g", dbg), ("db_fc", dbfc)):
        assert torch.equal(out[name], ref), name


@pytest.mark.gpu
def test_fused_chain_side_split_in_cuda_graph():
    """The side stream of the fused whole-backward call joins a CUDA graph capture and rejoins the
    captured stream: a replay gives the eager call's outputs bit for bit."""
    swg = _swg()
    shape = SwigluShape("split_M100000", 100000, 512, 1024, 12, "pages")
    inp = swiglu_inputs(shape, device="cuda")
    eager = swg.swiglu_bwd(**inp, fused=True, return_dg=False)
    swg.swg_check()
    out = {k: torch.empty_like(v) for k, v in eager.items()}
    ws = torch.empty(max(swg.swiglu_bwd_workspace_size(shape.M, shape.K, shape.N, swg.SWG_FUSED), 16), dtype=torch.uint8,
                     device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the call up outside the capture
        swg.swiglu_bwd(**inp, fused=True, return_dg=False, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        swg.swiglu_bwd(**inp, fused=True, return_dg=False, out=out, workspace=ws)
    for v in out.values():
        v.fill_(3.0e38)
    graph.replay()
    torch.cuda.synchronize()
    swg.swg_check()
    for k, v in eager.items():
        assert torch.equal(out[k], v), k
