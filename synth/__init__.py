"""Seeded synthetic workloads for the SwiGLU-FFN backward, SwishGrad and the
GroupNorm backward.

This package holds only input recipes (shapes, value distributions, seeds) and
the code that draws them. It contains none of the method's arithmetic, so both
the fp64 CPU oracle and the CUDA path can be fed from it without sharing any
computation.
"""

from .workloads import (  # noqa: F401
    GROUP_NORM_CONFIGS,
    GROUP_NORM_EPS,
    SWIGLU_CONFIGS,
    SWISH_CONFIG,
    SwigluShape,
    group_norm_inputs,
    swiglu_fwd_biases,
    swiglu_inputs,
    swish_inputs,
)
