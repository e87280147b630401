"""Randomised pins of the fp64 oracle on the CPU (hypothesis): the GroupNorm
backward against torch fp64 autograd of group_norm and against its eps = 0
invariants, and the activation gradients against torch fp64 autograd, over
random shapes, groupings and values."""

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402


@st.composite
def _gn_case(draw):
    G = draw(st.integers(1, 4))
    cg = draw(st.integers(1, 4))
    N = draw(st.integers(1, 3))
    S = draw(st.integers(1 if cg > 1 else 2, 9))  # torch's group_norm needs two values per group
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return N, G * cg, S, G, seed


@settings(max_examples=60, deadline=None, derandomize=True)
@given(_gn_case(), st.sampled_from([0.0, 1e-5, 1e-2]))
def test_group_norm_matches_torch_autograd(case, eps):
    import torch
    N, C, S, G, seed = case
    r = np.random.default_rng(seed)
    x = r.standard_normal((N, C, S)) * r.uniform(0.5, 3) + r.uniform(-3, 3)
    dy = r.standard_normal((N, C, S))
    gamma = 1.0 + 0.5 * r.standard_normal(C)
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    bt = torch.zeros(C, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.group_norm(xt, G, gt, bt, eps).backward(torch.tensor(dy))
    dx, dg, db = oracle.group_norm_bwd(dy, x, gamma, G, eps)
    scale = max(1.0, float(np.max(np.abs(dx))))
    assert np.max(np.abs(dx - xt.grad.numpy())) <= 1e-9 * scale
    assert np.max(np.abs(dg - gt.grad.numpy())) <= 1e-9 * max(1.0, float(np.max(np.abs(dg))))
    assert np.max(np.abs(db - bt.grad.numpy())) <= 1e-9 * max(1.0, float(np.max(np.abs(db))))
    if eps == 0.0:
        xg = x.reshape(N, G, -1)
        d = dx.reshape(N, G, -1)
        assert np.max(np.abs(d.sum(axis=2))) <= 1e-9 * scale * d.shape[2]
        assert np.max(np.abs((d * (xg - xg.mean(axis=2, keepdims=True))).sum(axis=2))) <= 1e-8 * scale * d.shape[2]


@settings(max_examples=40, deadline=None, derandomize=True)
@given(st.integers(0, 2 ** 31 - 1), st.sampled_from(["silu", "gelu", "hardswish"]))
def test_activation_gradients_match_torch_autograd(seed, act):
    import torch
    r = np.random.default_rng(seed)
    x = r.standard_normal(257) * r.uniform(0.1, 8)
    g = r.standard_normal(257)
    xt = torch.tensor(x, requires_grad=True)
    f = {"silu": torch.nn.functional.silu, "gelu": torch.nn.functional.gelu,
         "hardswish": torch.nn.functional.hardswish}[act]
    f(xt).backward(torch.tensor(g))
    assert np.max(np.abs(oracle.act_grad(g, x, act) - xt.grad.numpy())) <= 1e-12 * max(1.0, float(np.max(np.abs(g))))
