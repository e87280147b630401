"""The whole fused backward from host buffers (swiglu_bwd_host) vs the fp64
oracle and vs the device-resident call (GPU).

dx of every row is the same arithmetic as in the device-resident fused call,
so it must be bit-identical; dw and db come from fp32 partials split over
chunks and M-splits instead of M-splits alone, so they are compared with the
oracle under the usual contract (the w stage fed the chain's own bf16 dg, dfc,
which the device call returns, plus norm checks against the oracle's own
chain) and with the device call within one bf16 rounding.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import SWIGLU_CONFIGS, SwigluShape, swiglu_inputs

from ._parity import assert_all, compare, to_f64

pytestmark = pytest.mark.gpu


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _host_call(inp):
    swg = _swg()
    host = {k: v.cpu().pin_memory() for k, v in inp.items()}
    out = swg.swiglu_bwd_host(**host)
    torch.cuda.synchronize()
    swg.swg_check()
    return out


def _norm_only(rep, suffix):
    rep["ok"] = rep["finite"] and rep["max_err"] <= 2.0 ** -6 * rep["max_ref"] and rep["rel_l2"] <= 2.0 ** -8
    rep["name"] += suffix
    return rep


def _within_one_rounding(a, b):
    """|a - b| <= 2^-7 max(|a|, |b|) elementwise (one bf16 ulp), or both tiny."""
    a, b = to_f64(a), to_f64(b)
    return bool(np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-6))


def _case(shape: SwigluShape, full_oracle: bool):
    swg = _swg()
    inp = swiglu_inputs(shape, device="cuda")
    out = _host_call(inp)
    dev = swg.swiglu_bwd(**inp, fused=True, return_dg=True)
    torch.cuda.synchronize()
    assert torch.equal(out["dx"], dev["dx"].cpu()), "dx differs from the device-resident call"
    for k in ("dw_g", "dw_fc", "db_g", "db_fc"):
        assert _within_one_rounding(out[k], dev[k].cpu()), f"{k} differs from the device-resident call"
    h = {k: to_f64(v) for k, v in inp.items()}
    _, _, rdbg, rdbfc = oracle.swiglu_bwd_b(h["dy"], h["g"], h["fc"])
    reps = [compare("db_g", out["db_g"], rdbg), compare("db_fc", out["db_fc"], rdbfc)]
    gdg, gdfc = to_f64(dev["dg"]), to_f64(dev["dfc"])
    rdwg, rdwfc = oracle.swiglu_bwd_w(h["x"], gdg, gdfc)
    reps += [compare("dw_g", out["dw_g"], rdwg), compare("dw_fc", out["dw_fc"], rdwfc)]
    if full_oracle:
        rdx = oracle.swiglu_bwd_x(gdg, gdfc, h["w_g"], h["w_fc"])
        reps.append(compare("dx", out["dx"], rdx))
        ref = oracle.swiglu_bwd(h["x"], h["w_g"], h["w_fc"], h["dy"], h["g"], h["fc"], stage_dtype="bf16")
        for k in ("dw_g", "dw_fc", "dx"):
            reps.append(_norm_only(compare(k, out[k], ref[k]), "(oracle chain)"))
    return reps


def test_host_path_tiny_single_chunk():
    assert_all(_case(SWIGLU_CONFIGS["tiny"][0], full_oracle=True))


@pytest.mark.parametrize("M", [40000, 70001])
def test_host_path_chunked(M):
    # 40000 rows: one chunk (below two chunk sizes); 70001: two chunks, the last one ragged
    assert_all(_case(SwigluShape(f"host_M{M}", M, 512, 1024, 0, "pages"), full_oracle=True))


def test_host_path_pages_shape():
    # six chunks at the pages' shape: dx bit-identical to the device call, dw/db by the contract
    assert_all(_case(SWIGLU_CONFIGS["pages"][0], full_oracle=False))


def test_host_path_empty_M_writes_zero_sums():
    swg = _swg()
    K, N = 64, 128
    z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16).pin_memory()
    r = lambda *s: torch.randn(*s).to(torch.bfloat16).pin_memory()
    out = {k: torch.full(s, 3.0, dtype=torch.bfloat16).pin_memory()
           for k, s in (("dx", (0, K)), ("dw_g", (K, N)), ("dw_fc", (K, N)), ("db_g", (1, N)), ("db_fc", (1, N)))}
    swg.swiglu_bwd_host(z(0, K), r(K, N), r(K, N), z(0, N), z(0, N), z(0, N), out=out)
    torch.cuda.synchronize()
    for k in ("dw_g", "dw_fc", "db_g", "db_fc"):
        assert torch.count_nonzero(out[k]).item() == 0, k


def test_host_path_twice_in_a_row_is_deterministic():
    inp = swiglu_inputs(SwigluShape("host_M70001", 70001, 512, 1024, 0, "pages"), device="cuda")
    a = _host_call(inp)
    b = _host_call(inp)
    for k in a:
        assert torch.equal(a[k], b[k]), k
