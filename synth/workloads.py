"""Input recipes for the five workloads of the SwiGLU-FFN backward and SwishGrad.

Shapes and distributions follow the PyPTO-Gym fused SwiGLU backward walk-through
("Kernel signatures" and "Test cases" sections: dy, g, fc as [M, N], x as
[M, K], w_g and w_fc as [K, N], bf16, inputs scaled by 1/sqrt(M) and weights
by 1/sqrt(K), seed 0) and the CANN SwishGrad walk-through (grad and x of one
shape and dtype, fp32/fp16/bf16, float scale beta).

Reading of "N(0, s)": s is the standard deviation (values are randn * s),
because the tail-sweep workload is meant to drive sigma(g) into saturation,
which needs |g| well above 1.

Draw order for the SwiGLU workloads: x, w_g, w_fc, g, fc, dy, each as fp32
randn from one generator seeded with the workload's seed, multiplied by its
scale, then rounded to bf16 (round-to-nearest-even, torch's conversion).
SwishGrad draws x then grad, in fp32, then converts to the I/O dtype.

GroupNorm backward (the Ascend C backward blog post: an SD v1.5 UNet at
batch 2 and 512 x 512, whose largest GroupNorm input is [2, 320, 64, 64] with
32 groups, and ResNet-50 with GroupNorm, whose stage-1 activations at batch 32
are [32, 256, 56, 56]; fp16 in the post's kernel): per (sample, group) a mean
drawn from U(-2, 2) and a spread from U(0.5, 2), x = mean + spread * randn;
dy = randn; gamma = 1 + 0.5 randn; eps 1e-5. Draw order: the per-group means,
spreads, x's randn, dy, gamma, in fp32, then converted to the I/O dtype.

The generator device is a parameter: the CPU and CUDA generators give
different streams for the same seed, so a caller that compares two
implementations must feed both from ONE draw (draw once, copy to the other
side). Nothing here computes any part of the backward pass.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class SwigluShape:
    name: str
    M: int
    K: int
    N: int
    seed: int
    # standard deviations (before the 1/sqrt scaling flags below)
    dist: str  # "pages" | "tail" | "llm"


# The SwiGLU workloads: a tiny case, the dynamic-M tail sweep, the pages'
# own test shape (M=220000, K=512, N=1024) and an LLM-FFN-scale shape.
SWIGLU_CONFIGS = {
    "tiny": [SwigluShape("tiny", 256, 64, 128, 0, "pages")],
    "tail": [SwigluShape(f"tail_M{m}", m, 512, 1024, 2, "tail")
             for m in (1, 127, 1025, 4097, 65537)],
    "pages": [SwigluShape("pages", 220000, 512, 1024, 0, "pages")],
    "llm": [SwigluShape("llm", 16384, 4096, 14336, 3, "llm")],
}

# SwishGrad: lengths 2^24 and 2^24+7, three dtypes, two scales, seed 1.
SWISH_CONFIG = {
    "n": (1 << 24, (1 << 24) + 7),
    "dtypes": (torch.float32, torch.float16, torch.bfloat16),
    "scales": (1.0, 1.702),
    "seed": 1,
}


def _scales(shape: SwigluShape) -> dict:
    M, K, N = shape.M, shape.K, shape.N
    inv_m = 1.0 / math.sqrt(max(M, 1))
    inv_k = 1.0 / math.sqrt(K)
    if shape.dist == "pages":
        return dict(x=inv_m, w_g=inv_k, w_fc=inv_k, g=inv_m, fc=inv_m, dy=inv_m)
    if shape.dist == "tail":
        return dict(x=inv_m, w_g=inv_k, w_fc=inv_k, g=3.0, fc=1.0, dy=1.0)
    if shape.dist == "llm":
        inv_n = 1.0 / math.sqrt(N)
        return dict(x=1.0, w_g=inv_k, w_fc=inv_k, g=2.0, fc=inv_n, dy=inv_n)
    raise ValueError(f"unknown distribution {shape.dist!r}")


def swiglu_inputs(shape: SwigluShape, device: str | torch.device = "cpu",
                  seed: int | None = None) -> dict:
    """Draw x, w_g, w_fc, g, fc, dy (bf16, contiguous) for one SwiGLU workload."""
    M, K, N = shape.M, shape.K, shape.N
    sc = _scales(shape)
    gen = torch.Generator(device=device)
    gen.manual_seed(shape.seed if seed is None else seed)
    dims = dict(x=(M, K), w_g=(K, N), w_fc=(K, N), g=(M, N), fc=(M, N), dy=(M, N))
    out = {}
    for name in ("x", "w_g", "w_fc", "g", "fc", "dy"):
        t = torch.randn(dims[name], generator=gen, device=device, dtype=torch.float32)
        t.mul_(sc[name])
        out[name] = t.to(torch.bfloat16)
        del t
    return out


def swiglu_fwd_biases(shape: SwigluShape, device: str | torch.device = "cpu",
                      seed: int | None = None) -> tuple:
    """Draw the forward's biases (b_g, b_fc) [N] bf16, with the standard deviation
    of x W (the x scale: each product sums K terms of variance x^2 / K), from a
    generator seeded with the workload's seed + 1000 (independent of
    swiglu_inputs' draws)."""
    N = shape.N
    std = _scales(shape)["x"]
    gen = torch.Generator(device=device)
    gen.manual_seed((shape.seed if seed is None else seed) + 1000)
    b = [torch.randn(N, generator=gen, device=device, dtype=torch.float32).mul_(std).to(torch.bfloat16)
         for _ in range(2)]
    return b[0], b[1]


GROUP_NORM_CONFIGS = {
    # name: (N, C, HxW, G)
    "tiny": (2, 8, 12, 4),
    "sd_unet_64x64": (2, 320, 64 * 64, 32),
    "resnet50_stage1_b32": (32, 256, 56 * 56, 32),
    "vae_512x512": (1, 128, 512 * 512, 32),
}
GROUP_NORM_EPS = 1e-5


def group_norm_inputs(N: int, C: int, HxW: int, G: int, dtype: torch.dtype,
                      device: str | torch.device = "cpu", seed: int = 3) -> tuple:
    """Draw (dy, x, gamma) for the GroupNorm backward, x and dy as [N, C, HxW]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    mean = torch.rand(N, G, 1, generator=gen, device=device).mul_(4.0).sub_(2.0)
    spread = torch.rand(N, G, 1, generator=gen, device=device).mul_(1.5).add_(0.5)
    x = torch.randn(N, G, (C // G) * HxW, generator=gen, device=device).mul_(spread).add_(mean)
    dy = torch.randn(N, C, HxW, generator=gen, device=device)
    gamma = torch.randn(C, generator=gen, device=device).mul_(0.5).add_(1.0)
    return dy.to(dtype), x.reshape(N, C, HxW).to(dtype), gamma.to(dtype)


def swish_inputs(n: int, dtype: torch.dtype, device: str | torch.device = "cpu",
                 seed: int = 1) -> tuple:
    """Draw (grad, x) for SwishGrad: x ~ randn*4 (std 4), grad ~ randn."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(4.0)
    grad = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    return grad.to(dtype), x.to(dtype)
