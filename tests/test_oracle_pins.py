"""The fp64 oracle against facts that do not come from it (CPU only).

Also plants plausible mistakes in the oracle (on the CPU, via monkeypatch)
and checks that at least one pin catches each of them.
"""

import numpy as np
import pytest

import oracle.activations as oact
import oracle.group_norm as ogn
import oracle.numerics as onum
import oracle.swiglu as osw
import oracle.swish as osh

from . import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def _sig_wrong_sign(z):
    z = np.asarray(z, np.float64)
    return 1.0 / (1.0 + np.exp(np.clip(z, -700, 700)))


def _silu_grad_drop_term(z):
    s = osw.sigmoid(z)
    return s * (1.0 + z)


def _b_drop_fc(dy, g, fc):
    dy, g, fc = (np.asarray(a, np.float64) for a in (dy, g, fc))
    s = osw.sigmoid(g)
    dg = dy * (s * (1.0 + g * (1.0 - s)))
    dfc = dy * g * s
    return dg, dfc, dg.sum(0, keepdims=True), dfc.sum(0, keepdims=True)


def _b_dfc_sigma_only(dy, g, fc):
    dy, g, fc = (np.asarray(a, np.float64) for a in (dy, g, fc))
    s = osw.sigmoid(g)
    dg = dy * fc * (s * (1.0 + g * (1.0 - s)))
    dfc = dy * s
    return dg, dfc, dg.sum(0, keepdims=True), dfc.sum(0, keepdims=True)


def _b_db_mean(dy, g, fc):
    dg, dfc, _, _ = osw.__dict__["_orig_b"](dy, g, fc)
    return dg, dfc, dg.mean(0, keepdims=True), dfc.mean(0, keepdims=True)


def _w_swapped(x, dg, dfc):
    xt = np.asarray(x, np.float64).T
    return xt @ np.asarray(dfc, np.float64), xt @ np.asarray(dg, np.float64)


def _x_drop_fc_term(dg, dfc, w_g, w_fc):
    return np.asarray(dg, np.float64) @ np.asarray(w_g, np.float64).T


def _x_wrong_sign(dg, dfc, w_g, w_fc):
    return (np.asarray(dg, np.float64) @ np.asarray(w_g, np.float64).T
            - np.asarray(dfc, np.float64) @ np.asarray(w_fc, np.float64).T)


def _swish_no_beta_inside(grad, x, scale=1.0):
    x = np.asarray(x, np.float64)
    t = x
    s = osw.sigmoid(float(np.float32(scale)) * x)
    return np.asarray(grad, np.float64) * (s * (1.0 + t * (1.0 - s)))


def _swish_beta_not_f32(grad, x, scale=1.0):
    x = np.asarray(x, np.float64)
    b = 1.0 if scale is None else float(scale)
    t = b * x
    s = osw.sigmoid(t)
    return np.asarray(grad, np.float64) * (s * (1.0 + t * (1.0 - s)))


def _fwd_drops_bias_g(x, w_g, w_fc, b_g=None, b_fc=None):
    return osw.__dict__["_orig_fwd"](x, w_g, w_fc, None, b_fc)


def _fwd_sigmoid_not_silu(x, w_g, w_fc, b_g=None, b_fc=None):
    g, fc, _ = osw.__dict__["_orig_fwd"](x, w_g, w_fc, b_g, b_fc)
    return g, fc, osw.sigmoid(g) * fc


def _fwd_weights_swapped(x, w_g, w_fc, b_g=None, b_fc=None):
    return osw.__dict__["_orig_fwd"](x, w_fc, w_g, b_g, b_fc)


def _gelu_drops_x_phi(grad, x):
    from scipy.special import erf
    x = np.asarray(x, np.float64)
    return np.asarray(grad, np.float64) * 0.5 * (1.0 + erf(x / np.sqrt(2.0)))


def _hardswish_slope_sixth(grad, x):
    x = np.asarray(x, np.float64)
    return np.asarray(grad, np.float64) * np.where(x <= -3.0, 0.0, np.where(x < 3.0, x / 6.0 + 0.5, 1.0))


def _hardswish_kinks_closed(grad, x):
    x = np.asarray(x, np.float64)
    return np.asarray(grad, np.float64) * np.where(x < -3.0, 0.0, np.where(x <= 3.0, x / 3.0 + 0.5, 1.0))


def _gn_parts(dy, x, gamma, G, eps):
    dy, x = np.asarray(dy, np.float64), np.asarray(x, np.float64)
    N, C, S = x.shape
    g = np.ones(C) if gamma is None else np.asarray(gamma, np.float64)
    mu, _, rstd = ogn.group_norm_stats(x, G, eps)
    xhat = (x.reshape(N, G, -1) - mu[:, :, None]) * rstd[:, :, None]
    gdy = (dy * g[None, :, None]).reshape(N, G, -1)
    return dy, x, N, C, S, g, rstd, xhat, gdy


def _gn_drops_mean_term(dy, x, gamma, G, eps):
    dy, x, N, C, S, g, rstd, xhat, gdy = _gn_parts(dy, x, gamma, G, eps)
    m = xhat.shape[2]
    dx = rstd[:, :, None] * (gdy - xhat * (gdy * xhat).sum(2, keepdims=True) / m)
    return dx.reshape(N, C, S), (dy * xhat.reshape(N, C, S)).sum((0, 2)), dy.sum((0, 2))


def _gn_drops_xhat_term(dy, x, gamma, G, eps):
    dy, x, N, C, S, g, rstd, xhat, gdy = _gn_parts(dy, x, gamma, G, eps)
    m = xhat.shape[2]
    dx = rstd[:, :, None] * (gdy - gdy.sum(2, keepdims=True) / m)
    return dx.reshape(N, C, S), (dy * xhat.reshape(N, C, S)).sum((0, 2)), dy.sum((0, 2))


def _gn_gamma_outside_sums(dy, x, gamma, G, eps):
    dy, x, N, C, S, g, rstd, xhat, gdy = _gn_parts(dy, x, gamma, G, eps)
    m = xhat.shape[2]
    gc = np.repeat(g.reshape(G, -1), S, axis=1)[None]  # gamma of each element, [1, G, m]
    d = dy.reshape(N, G, -1)
    dx = rstd[:, :, None] * gc * (d - d.sum(2, keepdims=True) / m - xhat * (d * xhat).sum(2, keepdims=True) / m)
    return dx.reshape(N, C, S), (dy * xhat.reshape(N, C, S)).sum((0, 2)), dy.sum((0, 2))


def _gn_var_without_eps_in_last_term(dy, x, gamma, G, eps):
    dx, dgamma, dbeta = ogn.__dict__["_orig_gn"](dy, x, gamma, G, eps)
    dy_, x_, N, C, S, g, rstd, xhat, gdy = _gn_parts(dy, x, gamma, G, eps)
    m = xhat.shape[2]
    mu, var, _ = ogn.group_norm_stats(x_, G, eps)
    xc = x_.reshape(N, G, -1) - mu[:, :, None]
    last_ok = xhat * (gdy * xhat).sum(2, keepdims=True) / m
    with np.errstate(divide="ignore", invalid="ignore"):  # var = 0 in the one-element groups
        last_bad = xc * (gdy * xc).sum(2, keepdims=True) / (m * var[:, :, None])
    return dx + (rstd[:, :, None] * (last_ok - last_bad)).reshape(N, C, S), dgamma, dbeta


def _gn_dgamma_without_xhat(dy, x, gamma, G, eps):
    dx, _, dbeta = ogn.__dict__["_orig_gn"](dy, x, gamma, G, eps)
    return dx, dbeta.copy(), dbeta


def _gn_unbiased_var(x, G, eps):
    xg = np.asarray(x, np.float64).reshape(x.shape[0], G, -1)
    mu = xg.mean(axis=2)
    var = xg.var(axis=2, ddof=1)
    return mu, var, 1.0 / np.sqrt(var + eps)


def _bf16_truncate(x):
    v = np.asarray(x, np.float64).astype(np.float32)
    return ((v.view(np.uint32) >> 16) << 16).view(np.float32).astype(np.float64)


MUTANTS = {
    "sigmoid_sign": [(osw, "sigmoid", _sig_wrong_sign), (osh, "sigmoid", _sig_wrong_sign)],
    "silu_grad_drops_1_minus_s": [(osw, "silu_grad", _silu_grad_drop_term)],
    "dg_drops_fc": [(osw, "swiglu_bwd_b", _b_drop_fc)],
    "dfc_sigma_only": [(osw, "swiglu_bwd_b", _b_dfc_sigma_only)],
    "db_mean_not_sum": [(osw, "swiglu_bwd_b", _b_db_mean)],
    "dw_outputs_swapped": [(osw, "swiglu_bwd_w", _w_swapped)],
    "dx_drops_fc_term": [(osw, "swiglu_bwd_x", _x_drop_fc_term)],
    "dx_wrong_sign": [(osw, "swiglu_bwd_x", _x_wrong_sign)],
    "swish_beta_missing_in_bracket": [(osh, "swish_grad", _swish_no_beta_inside)],
    "swish_beta_not_rounded_to_f32": [(osh, "swish_grad", _swish_beta_not_f32)],
    "bf16_truncates": [(onum, "f64_to_bf16_value", _bf16_truncate)],
    "fwd_drops_bias_g": [(osw, "swiglu_fwd", _fwd_drops_bias_g)],
    "fwd_sigmoid_not_silu": [(osw, "swiglu_fwd", _fwd_sigmoid_not_silu)],
    "fwd_weights_swapped": [(osw, "swiglu_fwd", _fwd_weights_swapped)],
    "gelu_drops_x_phi": [(oact, "gelu_grad", _gelu_drops_x_phi)],
    "hardswish_slope_one_sixth": [(oact, "hardswish_grad", _hardswish_slope_sixth)],
    "hardswish_kinks_closed": [(oact, "hardswish_grad", _hardswish_kinks_closed)],
    "gn_drops_mean_term": [(ogn, "group_norm_bwd", _gn_drops_mean_term)],
    "gn_drops_xhat_term": [(ogn, "group_norm_bwd", _gn_drops_xhat_term)],
    "gn_gamma_outside_sums": [(ogn, "group_norm_bwd", _gn_gamma_outside_sums)],
    "gn_var_without_eps_in_last_term": [(ogn, "group_norm_bwd", _gn_var_without_eps_in_last_term)],
    "gn_dgamma_without_xhat": [(ogn, "group_norm_bwd", _gn_dgamma_without_xhat)],
    "gn_unbiased_var": [(ogn, "group_norm_stats", _gn_unbiased_var)],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    monkeypatch.setitem(osw.__dict__, "_orig_b", osw.swiglu_bwd_b)
    monkeypatch.setitem(osw.__dict__, "_orig_fwd", osw.swiglu_fwd)
    monkeypatch.setitem(ogn.__dict__, "_orig_gn", ogn.group_norm_bwd)
    for mod, attr, fn in MUTANTS[name]:
        monkeypatch.setattr(mod, attr, fn)
    caught = []
    for pin in _pins.ALL_PINS:
        try:
            pin()
        except Exception as e:  # AssertionError, or a shape error from a bad transpose
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught the planted mistake {name}"
