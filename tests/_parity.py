"""Comparison of CUDA-path outputs with the fp64 oracle.

Tolerances (element-wise |gpu - ref| <= atol + rtol * |ref|, ref = the
oracle's fp64 value rounded once to the output dtype):
  * dg, dfc, grad_x: rtol 2^-7, atol 1e-4 -- the SwiGLU backward walk-through's
    own assert_allclose tolerances ("Precision check" section);
  * db, dw, dx: rtol 2^-7, atol 1e-3.
Because those absolute tolerances can exceed the outputs' own magnitude at
small scales (an all-zero output would pass at the pages' shape), every
comparison also applies a scale-aware check:
  max|gpu - ref| <= 2^-6 * max|ref|   and   ||gpu - ref||_2 <= 2^-8 * ||ref||_2.
The relative-L2 part applies to tensors of at least L2_MIN_N elements: on a
handful of elements a single bf16 rounding that falls on the other side of a
tie from the oracle's (one ulp, up to 2^-7 of the value, which the
element-wise contract allows) can by itself exceed 2^-8 of the norm.
"""

from __future__ import annotations

import numpy as np

from oracle import round_to_dtype

RTOL = 2.0 ** -7
ATOL_ELEM = 1e-4
ATOL_RED = 1e-3
MAX_REL = 2.0 ** -6
L2_REL = 2.0 ** -8
L2_MIN_N = 64

ATOL = dict(dg=ATOL_ELEM, dfc=ATOL_ELEM, grad_x=ATOL_ELEM,
            db_g=ATOL_RED, db_fc=ATOL_RED, dw_g=ATOL_RED, dw_fc=ATOL_RED, dx=ATOL_RED,
            g=ATOL_RED, fc=ATOL_RED, y=ATOL_RED)  # forward: GEMM outputs, like dw and dx


def to_f64(t) -> np.ndarray:
    """torch tensor (any device, bf16/f16/f32) -> fp64 numpy, exactly."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(name: str, got, ref, dtype: str = "bf16", atol: float | None = None,
            scale_aware: bool = True) -> dict:
    """Return a report dict; 'ok' is True when every check passes."""
    g = to_f64(got) if not isinstance(got, np.ndarray) else np.asarray(got, np.float64)
    r = round_to_dtype(np.asarray(ref, np.float64), dtype)
    g = g.reshape(r.shape)
    atol = ATOL[name] if atol is None else atol
    rep = dict(name=name, n=int(r.size))
    if r.size == 0:
        rep.update(ok=True)
        return rep
    finite = bool(np.all(np.isfinite(g)))
    err = np.abs(g - r)
    bound = atol + RTOL * np.abs(r)
    bad = int(np.count_nonzero(~(err <= bound)))
    rmax = float(np.max(np.abs(r)))
    rl2 = float(np.linalg.norm(r))
    emax = float(np.max(err)) if finite else float("inf")
    el2 = float(np.linalg.norm(err)) if finite else float("inf")
    ok = finite and bad == 0
    if scale_aware and rmax > 0:
        ok = ok and emax <= MAX_REL * rmax and (r.size < L2_MIN_N or el2 <= L2_REL * rl2)
    rep.update(ok=ok, finite=finite, bad=bad, max_err=emax, max_ref=rmax,
               rel_l2=(el2 / rl2 if rl2 > 0 else 0.0))
    return rep


def assert_all(reports) -> None:
    failed = [r for r in reports if not r["ok"]]
    assert not failed, "parity failures:\n" + "\n".join(str(r) for r in failed)
