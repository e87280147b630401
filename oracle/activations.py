"""fp64 oracle of the sibling activation gradients (test infrastructure only).

Source: the Ascend C blog post on hand-written backward operators (its
closing recommendations name GELU and HardSwish as the next activations to
give a hand-written backward), and "SwishGrad in CANN ops-nn: principle,
implementation and the aclnnSwishBackward guide", whose closing section names
SiluGrad as a sibling of SwishGrad. Neither page prints these formulas; the
standard definitions are used, each as grad_x = grad * f'(x):

* SiLU:      f(x) = x sigma(x)                -> SwishGrad with beta = 1
* GELU:      f(x) = x Phi(x), exact (erf) form, Phi(x) = (1 + erf(x / sqrt 2)) / 2
             f'(x) = Phi(x) + x phi(x),  phi(x) = exp(-x^2 / 2) / sqrt(2 pi)
* HardSwish: f(x) = x min(max(x + 3, 0), 6) / 6
             f'(x) = 0 for x <= -3, x / 3 + 1/2 for -3 < x < 3, 1 for x >= 3
             (at the kinks the outer branches are taken, as PyTorch's autograd does)

Library primitives used as steps: scipy.special.erf, numpy.exp.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

from .swish import swish_grad

_INV_SQRT2 = 1.0 / math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def silu_act_grad(grad, x) -> np.ndarray:
    """grad * SiLU'(x): SwishGrad with beta = 1."""
    return swish_grad(grad, x, 1.0)


def gelu_grad(grad, x) -> np.ndarray:
    """grad * (Phi(x) + x phi(x))."""
    grad = np.asarray(grad, np.float64)
    x = np.asarray(x, np.float64)
    cdf = 0.5 * (1.0 + erf(x * _INV_SQRT2))
    pdf = _INV_SQRT_2PI * np.exp(-0.5 * x * x)
    return grad * (cdf + x * pdf)


def hardswish_grad(grad, x) -> np.ndarray:
    """grad * HardSwish'(x), the middle branch open at -3 and 3."""
    grad = np.asarray(grad, np.float64)
    x = np.asarray(x, np.float64)
    d = np.where(x <= -3.0, 0.0, np.where(x < 3.0, x / 3.0 + 0.5, 1.0))
    return grad * d


def act_grad(grad, x, act: str) -> np.ndarray:
    """Dispatch by name: "silu", "gelu" or "hardswish"."""
    return {"silu": silu_act_grad, "gelu": gelu_grad, "hardswish": hardswish_grad}[act](grad, x)
