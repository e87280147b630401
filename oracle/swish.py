"""fp64 oracle of SwishGrad (test infrastructure only).

Source: "SwishGrad in CANN ops-nn: principle, implementation and the
aclnnSwishBackward guide" (bhfrc.com/news/37500).

Section 1.2 ("Computation formula"): the forward is s(x) = x sigma(beta x);
its derivative is s'(x) = sigma(beta x) (1 + beta x (1 - sigma(beta x)));
the output is grad_x = grad * s'(x). The printed first form of s'(x) is
garbled by extraction; the second form, and the kernel's operation chain in
section 2.4 (beta*x -> negate -> exp -> +1 -> divide -> 1 - sigma -> times
beta x -> +1 -> times sigma -> times grad), agree with the line above.

Section 2.4: fp16/bf16 inputs are widened to fp32 and the result is narrowed
with round-to-nearest-even; fp32 stays fp32. Section 3.5: beta is carried
as a float and is 1.0 when absent. The oracle therefore uses beta's fp32
value, widened exactly, and computes everything else in fp64; the caller
rounds the result once to the I/O dtype.
"""

from __future__ import annotations

import numpy as np

from .swiglu import sigmoid


def _beta(scale) -> float:
    return 1.0 if scale is None else float(np.float32(scale))


def swish_fwd(x, scale=1.0) -> np.ndarray:
    """s(x) = x * sigma(beta x) (section 1.2), used only by the pins."""
    x = np.asarray(x, np.float64)
    return x * sigmoid(_beta(scale) * x)


def swish_grad(grad, x, scale=1.0) -> np.ndarray:
    """grad_x = grad * sigma(beta x) * (1 + beta x (1 - sigma(beta x)))."""
    grad = np.asarray(grad, np.float64)
    x = np.asarray(x, np.float64)
    t = _beta(scale) * x
    s = sigmoid(t)
    return grad * (s * (1.0 + t * (1.0 - s)))
