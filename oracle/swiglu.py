"""fp64 oracle of the SwiGLU-FFN backward (test infrastructure only).

Source: "PyPTO-Gym in practice: the fused SwiGLU backward operator"
(hnwysp.cn/news/34787).

Forward ("Operator background"):   Gate = x W_g + b_g,  FC = x W_fc + b_fc,
                                   y = SiLU(Gate) * FC,  SiLU(z) = z sigma(z).
Backward ("Algorithm overview and formulas", items 1-4), given upstream dy:
  1. dg  = dy * FC * SiLU'(g),  SiLU'(g) = sigma(g) (1 + g (1 - sigma(g)))
     dfc = dy * SiLU(g)       = dy * g * sigma(g)
  2. db_g = sum over the batch axis (rows) of dg;  db_fc likewise of dfc
  3. dw_g = x^T dg;  dw_fc = x^T dfc
  4. dx = dg W_g^T + dfc W_fc^T
Shapes ("Kernel signatures"): x [M, K]; w_g, w_fc [K, N]; dy, g, fc, dg, dfc
[M, N]; db_g, db_fc [1, N]; dw_g, dw_fc [K, N]; dx [M, K].

Readings where the page is garbled or silent:
* The printed formulas lost their "=", "+" and prime marks; the code
  paragraph under item 1 (dg = dy*fc * silu_bwd, dfc = dy * silu_g) fixes
  them as above.
* The page evaluates sigma as exp(g) / (1 + exp(g)); that form overflows
  for large g. Here sigma is evaluated in an overflow-free form that is the
  same function: 1/(1+exp(-z)) for z >= 0, exp(z)/(1+exp(z)) for z < 0.
* dw and dx consume dg and dfc. The three-kernel call chain passes them
  between kernels as bf16 tensors ("Kernel overview and call chain"), so
  `swiglu_bwd(..., stage_dtype="bf16")` rounds dg and dfc to bf16 before
  items 3-4; `stage_dtype=None` gives the exact gradient of the math.
"""

from __future__ import annotations

import numpy as np

from .numerics import round_to_dtype


def sigmoid(z) -> np.ndarray:
    """sigma(z) = 1 / (1 + e^-z), evaluated without overflow in fp64."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    e = np.exp(z[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def silu(z) -> np.ndarray:
    """SiLU(z) = z * sigma(z) ("Operator background")."""
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def silu_grad(z) -> np.ndarray:
    """SiLU'(z) = sigma(z) * (1 + z * (1 - sigma(z))) (item 1)."""
    z = np.asarray(z, dtype=np.float64)
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def swiglu_fwd(x, w_g, w_fc, b_g=None, b_fc=None):
    """Forward of the FFN gate ("Operator background"); returns (g, fc, y):
    g = x W_g + b_g, fc = x W_fc + b_fc, y = SiLU(g) * fc, in fp64.

    The reference for the forward kernel's parity tests; never an input
    producer for the backward's parity tests (those draw g, fc directly).
    """
    x = np.asarray(x, np.float64)
    g = x @ np.asarray(w_g, np.float64)
    fc = x @ np.asarray(w_fc, np.float64)
    if b_g is not None:
        g = g + np.asarray(b_g, np.float64).reshape(1, -1)
    if b_fc is not None:
        fc = fc + np.asarray(b_fc, np.float64).reshape(1, -1)
    return g, fc, silu(g) * fc


def swiglu_bwd_b(dy, g, fc):
    """b stage: dg, dfc [M, N] and db_g, db_fc [1, N] (items 1 and 2)."""
    dy = np.asarray(dy, np.float64)
    g = np.asarray(g, np.float64)
    fc = np.asarray(fc, np.float64)
    s = sigmoid(g)
    dg = dy * fc * (s * (1.0 + g * (1.0 - s)))
    dfc = dy * (g * s)
    db_g = dg.sum(axis=0, keepdims=True)
    db_fc = dfc.sum(axis=0, keepdims=True)
    return dg, dfc, db_g, db_fc


def swiglu_bwd_w(x, dg, dfc):
    """w stage: dw_g = x^T dg, dw_fc = x^T dfc, both [K, N] (item 3)."""
    xt = np.asarray(x, np.float64).T
    return xt @ np.asarray(dg, np.float64), xt @ np.asarray(dfc, np.float64)


def swiglu_bwd_x(dg, dfc, w_g, w_fc):
    """x stage: dx = dg W_g^T + dfc W_fc^T, [M, K] (item 4)."""
    return (np.asarray(dg, np.float64) @ np.asarray(w_g, np.float64).T
            + np.asarray(dfc, np.float64) @ np.asarray(w_fc, np.float64).T)


def swiglu_bwd(x, w_g, w_fc, dy, g, fc, stage_dtype: str | None = "bf16") -> dict:
    """The whole backward: b stage, then the w and x stages on its dg, dfc.

    stage_dtype="bf16": dg and dfc are rounded to bf16 before the w and x
    stages, as the call chain hands them over; None: exact math throughout.
    Returned dg, dfc, db are always the unrounded fp64 values.
    """
    dg, dfc, db_g, db_fc = swiglu_bwd_b(dy, g, fc)
    if stage_dtype is None:
        dg_s, dfc_s = dg, dfc
    else:
        dg_s, dfc_s = round_to_dtype(dg, stage_dtype), round_to_dtype(dfc, stage_dtype)
    dw_g, dw_fc = swiglu_bwd_w(x, dg_s, dfc_s)
    dx = swiglu_bwd_x(dg_s, dfc_s, w_g, w_fc)
    return dict(dg=dg, dfc=dfc, db_g=db_g, db_fc=db_fc, dw_g=dw_g, dw_fc=dw_fc, dx=dx)


def swiglu_bwd_sampled(x, w_g, w_fc, dy, g, fc, rows, cols,
                       stage_dtype: str | None = "bf16") -> dict:
    """Selected outputs of `swiglu_bwd`, for shapes too large to compute whole.

    rows: indices into M -> dg, dfc, dx at those rows (each dx row needs only
    its own dg, dfc row). cols: indices into N -> db_g, db_fc, dw_g, dw_fc at
    those columns (each needs only its own dg, dfc column over all M).
    Every sampled value is the same definition applied to a slice.
    Inputs may be torch tensors or numpy arrays; each slice is widened to fp64.
    """
    def f64(t):
        if hasattr(t, "double"):
            return t.double().numpy()
        return np.asarray(t, np.float64)

    rows = np.asarray(rows)
    cols = np.asarray(cols)
    out = {}
    dg_r, dfc_r, _, _ = swiglu_bwd_b(f64(dy[rows]), f64(g[rows]), f64(fc[rows]))
    out["dg"], out["dfc"] = dg_r, dfc_r
    if stage_dtype is not None:
        dg_r, dfc_r = round_to_dtype(dg_r, stage_dtype), round_to_dtype(dfc_r, stage_dtype)
    out["dx"] = swiglu_bwd_x(dg_r, dfc_r, f64(w_g), f64(w_fc))

    dg_c, dfc_c, db_g, db_fc = swiglu_bwd_b(f64(dy[:, cols]), f64(g[:, cols]), f64(fc[:, cols]))
    out["db_g"], out["db_fc"] = db_g, db_fc
    if stage_dtype is not None:
        dg_c, dfc_c = round_to_dtype(dg_c, stage_dtype), round_to_dtype(dfc_c, stage_dtype)
    out["dw_g"], out["dw_fc"] = swiglu_bwd_w(f64(x), dg_c, dfc_c)
    return out
