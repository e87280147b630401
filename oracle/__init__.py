"""fp64 CPU oracle for the SwiGLU-FFN backward and SwishGrad.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this package: only the tests, the package's smoke check and the benchmark's
CPU-baseline leg use it. It shares no code with the CUDA path.

It restates, in plain numpy float64, what two pages define:

* "PyPTO-Gym in practice: the fused SwiGLU backward operator"
  (hnwysp.cn/news/34787), section "Algorithm overview and formulas",
  items 1-4 (dg, dfc, db_g, db_fc, dw_g, dw_fc, dx), plus the forward in its
  "Operator background" section (g, fc, y).
* "SwishGrad in CANN ops-nn: principle, implementation and the
  aclnnSwishBackward guide" (bhfrc.com/news/37500), section 1.2
  "Computation formula" (grad_x = grad * sigma(beta x) * (1 + beta x (1 -
  sigma(beta x)))), section 2.4 (fp16/bf16 widened to fp32, results narrowed
  with round-to-nearest-even), section 3.5 (beta defaults to 1.0).
* The sibling activation gradients (SiLU, GELU, HardSwish) that the Ascend C
  backward blog post and the SwishGrad page name, with their standard
  definitions (the pages print no formula for them): `activations.py`.
* The GroupNorm backward of the Ascend C backward blog post (its GroupNorm
  section, both printed versions): dx by the post's formula, dgamma and dbeta
  by their standard definitions: `group_norm.py`.

Library primitives used as steps: numpy.exp, numpy matmul, numpy.sum, numpy.mean.
Parity status: every function here is pinned by the `-m "not gpu"` tests
(closed forms, symbolic derivatives, finite differences of the forward,
brute-force loops, torch fp64 autograd); none is "parity unpinned".
"""

from .numerics import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    f64_to_bf16_value,
    round_to_dtype,
)
from .swiglu import (  # noqa: F401
    sigmoid,
    silu,
    silu_grad,
    swiglu_bwd,
    swiglu_bwd_b,
    swiglu_bwd_sampled,
    swiglu_bwd_w,
    swiglu_bwd_x,
    swiglu_fwd,
)
from .swish import swish_fwd, swish_grad  # noqa: F401
from .activations import act_grad, gelu_grad, hardswish_grad, silu_act_grad  # noqa: F401
from .group_norm import group_norm_bwd, group_norm_fwd, group_norm_stats  # noqa: F401
