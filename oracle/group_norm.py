"""fp64 oracle of the GroupNorm backward (test infrastructure only).

Source: "Beyond automatic differentiation: efficient custom backward operators
in Ascend C" (the Ascend C backward blog post). Its GroupNorm section is
printed twice: the first version (section 3.1, forward recap; 3.2, simplified
backward formula; 3.3, implementation notes and per-group pseudocode) and the
revised version (section 3.1, the formula with gamma; 3.2, the two-pass
per-group strategy; 3.3, the per-group kernel).

Forward (both versions, 3.1): the channels of each sample are split into G
groups of C / G consecutive channels; with m = (C / G) * HxW elements in a
group,
    mu = mean(x_group),  var = mean((x_group - mu)^2)   (biased),
    x_hat = (x - mu) / sqrt(var + eps),  y = gamma_c * x_hat + beta_c.
Backward, dx (revised version 3.1; gamma inside the sums):
    dx_i = (1 / sqrt(var + eps)) * ( gamma_c dy_i - (1/m) sum_j gamma_cj dy_j
                                      - (x_hat_i / m) sum_j gamma_cj dy_j x_hat_j ).
The first version's formula is the same with gamma = 1; its pseudocode divides
the last term by m * var instead of m * (var + eps), read as a misprint (the
formula above it has var + eps, and only that form is the derivative).
The pages give only dx; the parameter gradients a GroupNorm backward also
returns are the standard ones:
    dgamma_c = sum over samples and positions of dy * x_hat,
    dbeta_c  = sum over samples and positions of dy.
The statistics are recomputed from x, as the pages' kernel does (it loads x and
dy and forms mu and var itself).

Layout: x, dy, dx are [N, C, HxW] (NCHW with the spatial dimensions
flattened); gamma, dgamma, dbeta are [C]. Library primitives used as steps:
numpy mean, sum, sqrt.
"""

from __future__ import annotations

import numpy as np


def _groups(a: np.ndarray, G: int) -> np.ndarray:
    """[N, C, HxW] -> [N, G, C/G, HxW] (a view: group g holds channels g*C/G ... (g+1)*C/G - 1)."""
    N, C, S = a.shape
    return a.reshape(N, G, C // G, S)


def group_norm_stats(x, G: int, eps: float):
    """Per (sample, group): mu, var (biased) and rstd = 1 / sqrt(var + eps), each [N, G]."""
    xg = _groups(np.asarray(x, np.float64), G)
    mu = xg.mean(axis=(2, 3))
    var = ((xg - mu[:, :, None, None]) ** 2).mean(axis=(2, 3))
    return mu, var, 1.0 / np.sqrt(var + eps)


def group_norm_fwd(x, gamma, beta, G: int, eps: float) -> np.ndarray:
    """y = gamma_c * (x - mu) / sqrt(var + eps) + beta_c (used by the pins' finite differences)."""
    x = np.asarray(x, np.float64)
    N, C, S = x.shape
    mu, _, rstd = group_norm_stats(x, G, eps)
    xhat = (_groups(x, G) - mu[:, :, None, None]) * rstd[:, :, None, None]
    g = np.ones(C) if gamma is None else np.asarray(gamma, np.float64)
    b = np.zeros(C) if beta is None else np.asarray(beta, np.float64)
    return xhat.reshape(N, C, S) * g[None, :, None] + b[None, :, None]


def group_norm_bwd(dy, x, gamma, G: int, eps: float):
    """(dx, dgamma, dbeta) of GroupNorm; gamma None means all ones.

    dx follows the revised version's formula term by term: with gdy = gamma_c * dy,
    dx = rstd * (gdy - sum(gdy) / m - x_hat * sum(gdy * x_hat) / m), the sums over the group.
    """
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    N, C, S = x.shape
    if C % G != 0:
        raise ValueError("C must be a multiple of G")
    m = (C // G) * S
    g = np.ones(C) if gamma is None else np.asarray(gamma, np.float64)
    mu, _, rstd = group_norm_stats(x, G, eps)
    xhat = (_groups(x, G) - mu[:, :, None, None]) * rstd[:, :, None, None]  # [N, G, C/G, S]
    gdy = _groups(dy * g[None, :, None], G)
    sum_gdy = gdy.sum(axis=(2, 3))[:, :, None, None]
    sum_gdy_xhat = (gdy * xhat).sum(axis=(2, 3))[:, :, None, None]
    dx = rstd[:, :, None, None] * (gdy - sum_gdy / m - xhat * sum_gdy_xhat / m)
    dgamma = (dy * xhat.reshape(N, C, S)).sum(axis=(0, 2))
    dbeta = dy.sum(axis=(0, 2))
    return dx.reshape(N, C, S), dgamma, dbeta
