"""Exact widening and correctly rounded narrowing between fp64 and the I/O types.

Part of the fp64 oracle (test infrastructure only).

The SwiGLU backward walk-through stores every tensor as bf16 and computes in
fp32 ("Dtype conversion flow" section); the SwishGrad walk-through narrows
fp16/bf16 results with CAST_RINT, i.e. round-to-nearest-even (section 2.4).
The oracle keeps fp64 values and rounds ONCE, directly from fp64, to the
output type for comparison. Rounding fp64 -> fp32 -> bf16 would round twice
and can differ from this in the last bit, so bf16 narrowing is written out
from the format's definition (8 exponent bits, 7 stored mantissa bits).
"""

from __future__ import annotations

import numpy as np

_BF16_MAX = float.fromhex("0x1.fep127")      # largest finite bf16
_BF16_MIN_NORMAL_EXP = -126                   # 2**-126 is the smallest normal
_BF16_SUBNORMAL_ULP = 2.0 ** -133             # spacing below 2**-126


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16/int16 array) to fp64, exactly."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):          # NaN patterns widen to NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_value(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    Normal range: write |x| = m * 2**e with m in [0.5, 1); a bf16 significand
    has 8 bits, so the result is rint(m * 2**8) * 2**(e - 8), where numpy's
    rint rounds half to even. Below 2**-126 the spacing is fixed at 2**-133.
    Values whose rounded magnitude exceeds the largest bf16 become +-inf.
    NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    m, e = np.frexp(x)
    normal = np.abs(x) >= 2.0 ** _BF16_MIN_NORMAL_EXP
    out[normal] = np.ldexp(np.rint(m[normal] * 256.0), e[normal] - 8)
    sub = ~normal
    out[sub] = np.rint(x[sub] / _BF16_SUBNORMAL_ULP) * _BF16_SUBNORMAL_ULP
    big = np.abs(out) > _BF16_MAX
    out[big] = np.copysign(np.inf, x[big])
    out[np.isinf(x)] = x[np.isinf(x)]
    out[np.isnan(x)] = np.nan
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 to bf16 (ties to even) and return the uint16 bit patterns."""
    v = f64_to_bf16_value(x).astype(np.float32)     # exact: v is a bf16 value
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def round_to_dtype(x, dtype: str) -> np.ndarray:
    """Round fp64 values once to 'bf16', 'f16' or 'f32' and widen back to fp64.

    fp16 and fp32 use numpy's conversions, which round fp64 directly to the
    nearest representable value with ties to even.
    """
    x = np.asarray(x, dtype=np.float64)
    if dtype == "bf16":
        return f64_to_bf16_value(x)
    if dtype == "f16":
        return x.astype(np.float16).astype(np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "f64":
        return x
    raise ValueError(dtype)
