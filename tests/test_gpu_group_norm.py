"""GroupNorm backward through the C ABI vs the fp64 oracle (GPU).

dx is judged like the element-wise outputs (|gpu - ref| <= 1e-4 + 2^-7 |ref|),
dgamma and dbeta like the sums over rows (atol 1e-3), each ref the oracle's
fp64 value rounded once to the I/O dtype, plus the scale-aware checks. Inputs:
the GroupNorm recipe of synth/workloads.py (a different mean and spread per
group, gamma around 1).

Shapes cover both kernels and their load paths: the persistent
double-buffered kernel (16-byte aligned groups whose slices fit two buffers;
16-byte vectors, or scalar math when HxW is not a multiple of the vector;
one or several groups per cluster) and the one-group-per-cluster kernel
(slices longer than the shared-memory stage, read again for pass 2; plain
loads when a group does not start on 16 bytes); one to eight CTAs per group,
empty slices, one channel per group and one element per group.
"""

import numpy as np
import pytest
import torch

import oracle
from synth import GROUP_NORM_CONFIGS, GROUP_NORM_EPS, group_norm_inputs

from ._parity import ATOL_ELEM, ATOL_RED, assert_all, compare, to_f64

pytestmark = pytest.mark.gpu

DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
ALL_DT = list(DT)


def _swg():
    import swiglu_ffn_backward_gb300 as swg
    return swg


def _check(dy, x, gamma, G, eps, dx, dgamma, dbeta):
    ref_dx, ref_dg, ref_db = oracle.group_norm_bwd(
        to_f64(dy), to_f64(x), None if gamma is None else to_f64(gamma), G, eps)
    dt = DT[x.dtype]
    reps = [compare("gn_dx", dx, ref_dx, dtype=dt, atol=ATOL_ELEM)]
    if dgamma is not None:
        reps.append(compare("dgamma", dgamma, ref_dg, dtype=dt, atol=ATOL_RED))
        reps.append(compare("dbeta", dbeta, ref_db, dtype=dt, atol=ATOL_RED))
    return reps


def _run(shape, dtype, seed=5, gamma=True, params=True):
    N, C, HxW, G = shape
    dy, x, g = group_norm_inputs(N, C, HxW, G, dtype, device="cuda", seed=seed)
    g = g if gamma else None
    dx, dgamma, dbeta = _swg().group_norm_bwd(dy, x, G, gamma=g, eps=GROUP_NORM_EPS, params=params)
    torch.cuda.synchronize()
    _swg().swg_check()
    return _check(dy, x, g, G, GROUP_NORM_EPS, dx, dgamma, dbeta)


SMALL = [
    (2, 8, 12, 4),      # tiny; bulk + vectors in fp16/bf16 (m = 24), bulk scalar in fp32
    (3, 6, 49, 3),      # m = 98: plain loads in fp16/bf16, bulk scalar in fp32
    (2, 6, 4, 6),       # one channel per group
    (4, 5, 1, 5),       # one element per group (var = 0)
    (5, 12, 33, 4),     # m = 99: plain loads in every dtype
    (2, 64, 49, 32),    # 7 x 7 spatial
    (7, 10, 1000, 5),   # two channels per group, vector path
    (2, 1280, 64, 32),  # 40 channels per group, 8 x 8 spatial
    (2, 640, 1024, 32), # several CTAs per group
    (1, 4, 200000, 2),  # eight CTAs per group, slices longer than the stage
    (3, 9, 17, 3),      # ragged everything
    (1, 8, 20001, 1),   # streamed slices with scalar math (aligned groups, HxW not a vector multiple)
    (64, 32, 64, 32),   # 2048 small groups: each persistent cluster walks several of them
]


@pytest.mark.parametrize("dtype", ALL_DT, ids=lambda d: DT[d])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_group_norm_small_shapes(shape, dtype):
    assert_all(_run(shape, dtype))


@pytest.mark.parametrize("dtype", ALL_DT, ids=lambda d: DT[d])
def test_group_norm_sd_unet(dtype):
    assert_all(_run(GROUP_NORM_CONFIGS["sd_unet_64x64"], dtype))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=lambda d: DT[d])
def test_group_norm_resnet50_batch32(dtype):
    assert_all(_run(GROUP_NORM_CONFIGS["resnet50_stage1_b32"], dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=lambda d: DT[d])
def test_group_norm_large_groups_streamed(dtype):
    # 1M elements per group: eight CTAs, each reading its slice again for pass 2
    assert_all(_run(GROUP_NORM_CONFIGS["vae_512x512"], dtype))


@pytest.mark.parametrize("dtype", ALL_DT, ids=lambda d: DT[d])
def test_group_norm_without_gamma_and_dx_only(dtype):
    assert_all(_run((3, 16, 100, 4), dtype, gamma=False))
    assert_all(_run((3, 16, 100, 4), dtype, params=False))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16], ids=lambda d: DT[d])
def test_group_norm_misaligned_views(dtype):
    # tensors that start one element past a 16-byte boundary take the plain-load path
    swg = _swg()
    N, C, HxW, G = 2, 32, 256, 8
    dy, x, g = group_norm_inputs(N, C, HxW, G, dtype, device="cuda", seed=11)
    n = dy.numel()
    bdy = torch.empty(n + 1, dtype=dtype, device="cuda")
    bx = torch.empty(n + 1, dtype=dtype, device="cuda")
    bo = torch.empty(n + 1, dtype=dtype, device="cuda")
    bdy[1:].copy_(dy.reshape(-1))
    bx[1:].copy_(x.reshape(-1))
    vdy, vx, vo = bdy[1:].view(N, C, HxW), bx[1:].view(N, C, HxW), bo[1:].view(N, C, HxW)
    dx, dgamma, dbeta = swg.group_norm_bwd(vdy, vx, G, gamma=g, eps=GROUP_NORM_EPS, dx=vo)
    torch.cuda.synchronize()
    assert dx.data_ptr() == vo.data_ptr()
    assert_all(_check(dy, x, g, G, GROUP_NORM_EPS, dx, dgamma, dbeta))


def test_group_norm_is_deterministic():
    swg = _swg()
    N, C, HxW, G = GROUP_NORM_CONFIGS["sd_unet_64x64"]
    dy, x, g = group_norm_inputs(N, C, HxW, G, torch.float32, device="cuda", seed=12)
    a = swg.group_norm_bwd(dy, x, G, gamma=g)
    b = swg.group_norm_bwd(dy, x, G, gamma=g)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_group_norm_large_mean_fp32():
    # |mean| / spread ~ 100: the shifted sums keep the variance accurate
    swg = _swg()
    N, C, HxW, G = 2, 32, 1024, 8
    dy, x, g = group_norm_inputs(N, C, HxW, G, torch.float32, device="cuda", seed=13)
    x = x + 100.0
    out = swg.group_norm_bwd(dy, x, G, gamma=g, eps=GROUP_NORM_EPS)
    torch.cuda.synchronize()
    assert_all(_check(dy, x, g, G, GROUP_NORM_EPS, *out))


def test_group_norm_empty():
    swg = _swg()
    x = torch.empty(0, 8, 5, dtype=torch.bfloat16, device="cuda")
    dx, dgamma, dbeta = swg.group_norm_bwd(x, x, 4, gamma=torch.ones(8, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert dx.numel() == 0
    assert torch.count_nonzero(dgamma).item() == 0 and torch.count_nonzero(dbeta).item() == 0
    x = torch.empty(3, 8, 0, dtype=torch.float32, device="cuda")
    dx, dgamma, dbeta = swg.group_norm_bwd(x, x, 2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dgamma).item() == 0 and torch.count_nonzero(dbeta).item() == 0


def test_group_norm_dx_sums_to_zero_per_group():
    # the invariant the oracle pins (eps = 0 version) also holds for the kernel, up to rounding
    swg = _swg()
    N, C, HxW, G = 4, 32, 256, 8
    dy, x, g = group_norm_inputs(N, C, HxW, G, torch.float32, device="cuda", seed=14)
    dx, _, _ = swg.group_norm_bwd(dy, x, G, gamma=g, eps=0.0, params=False)
    torch.cuda.synchronize()
    s = to_f64(dx).reshape(N, G, -1).sum(axis=2)
    scale = np.abs(to_f64(dx)).max() * np.sqrt((C // G) * HxW)
    assert np.max(np.abs(s)) <= 1e-5 * scale
