"""Seeded synthetic workloads for the SwiGLU-FFN backward and SwishGrad.

This package holds only input recipes (shapes, value distributions, seeds) and
the code that draws them. It contains none of the method's arithmetic, so both
the fp64 CPU oracle and the CUDA path can be fed from it without sharing any
computation.
"""

from .workloads import (  # noqa: F401
    SWIGLU_CONFIGS,
    SWISH_CONFIG,
    SwigluShape,
    swiglu_fwd_biases,
    swiglu_inputs,
    swish_inputs,
)
