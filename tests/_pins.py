"""Pins of the fp64 oracle: checks against facts that do not come from the oracle.

Each pin raises AssertionError when the oracle disagrees with a closed form,
a symbolic derivative (sympy), a finite difference of a forward written out
here, a brute-force loop, an independent library routine (scipy.special.expit,
torch fp64 autograd, torch's bf16 conversion), or an invariant of the
mathematics. Functions are looked up on the oracle modules at call time, so a
test can plant a mistake in the oracle (monkeypatch) and check that some pin
catches it.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle.activations as oact
import oracle.group_norm as ogn
import oracle.numerics as onum
import oracle.swiglu as osw
import oracle.swish as osh

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=1234):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------- sigma

def pin_sigmoid_closed_forms():
    s = osw.sigmoid
    assert s(np.array([0.0]))[0] == 0.5
    # e^{-ln 3} = 1/3  ->  sigma(ln 3) = 3/4 ; sigma(-ln 3) = 1/4
    assert abs(s(np.array([math.log(3.0)]))[0] - 0.75) < 1e-15
    assert abs(s(np.array([-math.log(3.0)]))[0] - 0.25) < 1e-15
    z = np.linspace(-40, 40, 801)
    assert np.max(np.abs(s(z) + s(-z) - 1.0)) < 1e-15
    with np.errstate(over="raise", invalid="raise"):
        big = s(np.array([-1000.0, 1000.0, -745.0, 745.0]))
    assert big[0] == 0.0 and big[1] == 1.0 and 0.0 <= big[2] < 1e-300 and big[3] == 1.0


def pin_sigmoid_matches_scipy():
    from scipy.special import expit
    z = np.concatenate([np.linspace(-60, 60, 2401), _rng().standard_normal(1000) * 5])
    ref = expit(z)
    got = osw.sigmoid(z)
    assert np.all(np.abs(got - ref) <= 4e-16 * np.maximum(ref, 1e-300) + 1e-300)


def pin_sigmoid_derivative():
    z = np.linspace(-12, 12, 97)
    h = 1e-5
    fd = (osw.sigmoid(z + h) - osw.sigmoid(z - h)) / (2 * h)
    s = osw.sigmoid(z)
    # sigma' peaks at 1/4; truncation error ~h^2/24, rounding error ~1e-16/h
    assert np.max(np.abs(fd - s * (1 - s))) < 1e-9


# --------------------------------------------------------------------------- SiLU'

def _silu_local(z):
    # SiLU written out directly (z / (1 + e^-z)), independent of the oracle
    return z / (1.0 + np.exp(-z))


def pin_silu_grad_fd():
    z = np.linspace(-15, 15, 121)
    h = 1e-5 * np.maximum(1.0, np.abs(z))
    fd = (_silu_local(z + h) - _silu_local(z - h)) / (2 * h)
    got = osw.silu_grad(z)
    assert np.max(np.abs(fd - got)) < 1e-8


def pin_silu_grad_symbolic():
    import sympy as sp
    zs = sp.symbols("z")
    d = sp.diff(zs / (1 + sp.exp(-zs)), zs)
    pts = [-30.0, -7.5, -2.0, -0.3, 0.0, 0.25, 1.0, 3.5, 9.0, 30.0]
    ref = np.array([float(d.subs(zs, sp.Float(p, 40)).evalf(40)) for p in pts])
    got = osw.silu_grad(np.array(pts))
    assert np.all(np.abs(got - ref) <= 1e-14 * np.abs(ref) + 1e-300)


# --------------------------------------------------------------------------- b stage

def pin_b_stage_symbolic():
    import sympy as sp
    g_, fc_, dy_ = sp.symbols("g fc dy")
    y = g_ / (1 + sp.exp(-g_)) * fc_          # y = SiLU(g) * fc
    dg_e = dy_ * sp.diff(y, g_)
    dfc_e = dy_ * sp.diff(y, fc_)
    rng = _rng(7)
    G = rng.standard_normal(6) * 4
    FC = rng.standard_normal(6)
    DY = rng.standard_normal(6)
    dg, dfc, _, _ = osw.swiglu_bwd_b(DY[None, :], G[None, :], FC[None, :])
    for i in range(6):
        sub = {g_: sp.Float(G[i], 40), fc_: sp.Float(FC[i], 40), dy_: sp.Float(DY[i], 40)}
        rg = float(dg_e.subs(sub).evalf(40))
        rf = float(dfc_e.subs(sub).evalf(40))
        assert abs(dg[0, i] - rg) <= 1e-13 * abs(rg) + 1e-300
        assert abs(dfc[0, i] - rf) <= 1e-13 * abs(rf) + 1e-300


def pin_b_stage_fd():
    rng = _rng(11)
    M, N = 5, 7
    g = rng.standard_normal((M, N)) * 3
    fc = rng.standard_normal((M, N))
    dy = rng.standard_normal((M, N))
    dg, dfc, db_g, db_fc = osw.swiglu_bwd_b(dy, g, fc)
    h = 1e-6
    fd_g = dy * (_silu_local(g + h) * fc - _silu_local(g - h) * fc) / (2 * h)
    fd_fc = dy * (_silu_local(g) * (fc + h) - _silu_local(g) * (fc - h)) / (2 * h)
    assert np.max(np.abs(dg - fd_g)) < 1e-7
    assert np.max(np.abs(dfc - fd_fc)) < 1e-7
    assert db_g.shape == (1, N) and db_fc.shape == (1, N)


def pin_db_is_column_sum():
    rng = _rng(3)
    M, N = 9, 4
    dy, g, fc = (rng.standard_normal((M, N)) for _ in range(3))
    dg, dfc, db_g, db_fc = osw.swiglu_bwd_b(dy, g, fc)
    for n in range(N):
        sg = 0.0
        sf = 0.0
        for m in range(M):
            sg += dg[m, n]
            sf += dfc[m, n]
        assert abs(db_g[0, n] - sg) < 1e-13 and abs(db_fc[0, n] - sf) < 1e-13


# --------------------------------------------------------------------------- w, x stages

def pin_gemm_bruteforce():
    rng = _rng(5)
    M, K, N = 6, 3, 4
    x = rng.standard_normal((M, K))
    dg = rng.standard_normal((M, N))
    dfc = rng.standard_normal((M, N))
    w_g = rng.standard_normal((K, N))
    w_fc = rng.standard_normal((K, N))
    dw_g, dw_fc = osw.swiglu_bwd_w(x, dg, dfc)
    dx = osw.swiglu_bwd_x(dg, dfc, w_g, w_fc)
    assert dw_g.shape == (K, N) and dx.shape == (M, K)
    for k in range(K):
        for n in range(N):
            a = sum(x[m, k] * dg[m, n] for m in range(M))
            b = sum(x[m, k] * dfc[m, n] for m in range(M))
            assert abs(dw_g[k, n] - a) < 1e-12 and abs(dw_fc[k, n] - b) < 1e-12
    for m in range(M):
        for k in range(K):
            a = sum(dg[m, n] * w_g[k, n] + dfc[m, n] * w_fc[k, n] for n in range(N))
            assert abs(dx[m, k] - a) < 1e-12


# --------------------------------------------------------------------------- whole chain

def _loss_local(x, w_g, w_fc, b_g, b_fc, dy):
    g = x @ w_g + b_g
    fc = x @ w_fc + b_fc
    return float(np.sum(dy * _silu_local(g) * fc))


def pin_full_chain_fd():
    """Central differences of L = sum(dy * SiLU(x W_g + b_g) * (x W_fc + b_fc))."""
    rng = _rng(21)
    M, K, N = 4, 3, 5
    P = dict(x=rng.standard_normal((M, K)), w_g=rng.standard_normal((K, N)),
             w_fc=rng.standard_normal((K, N)), b_g=rng.standard_normal(N),
             b_fc=rng.standard_normal(N))
    dy = rng.standard_normal((M, N))
    g = P["x"] @ P["w_g"] + P["b_g"]
    fc = P["x"] @ P["w_fc"] + P["b_fc"]
    out = osw.swiglu_bwd(P["x"], P["w_g"], P["w_fc"], dy, g, fc, stage_dtype=None)
    want = dict(x="dx", w_g="dw_g", w_fc="dw_fc", b_g="db_g", b_fc="db_fc")
    h = 1e-6
    for pname, oname in want.items():
        fd = np.zeros_like(P[pname])
        for idx in np.ndindex(P[pname].shape):
            Pp = {k: v.copy() for k, v in P.items()}
            Pm = {k: v.copy() for k, v in P.items()}
            Pp[pname][idx] += h
            Pm[pname][idx] -= h
            fd[idx] = (_loss_local(dy=dy, **Pp) - _loss_local(dy=dy, **Pm)) / (2 * h)
        got = np.asarray(out[oname]).reshape(fd.shape)
        assert np.max(np.abs(got - fd)) < 1e-6, (oname, np.max(np.abs(got - fd)))


def pin_torch_autograd():
    import torch
    rng = _rng(33)
    M, K, N = 7, 6, 9
    x = torch.tensor(rng.standard_normal((M, K)), dtype=torch.float64, requires_grad=True)
    w_g = torch.tensor(rng.standard_normal((K, N)), dtype=torch.float64, requires_grad=True)
    w_fc = torch.tensor(rng.standard_normal((K, N)), dtype=torch.float64, requires_grad=True)
    b_g = torch.tensor(rng.standard_normal(N), dtype=torch.float64, requires_grad=True)
    b_fc = torch.tensor(rng.standard_normal(N), dtype=torch.float64, requires_grad=True)
    dy = torch.tensor(rng.standard_normal((M, N)), dtype=torch.float64)
    g = x @ w_g + b_g
    fc = x @ w_fc + b_fc
    y = torch.nn.functional.silu(g) * fc
    y.backward(dy)
    out = osw.swiglu_bwd(x.detach().numpy(), w_g.detach().numpy(), w_fc.detach().numpy(),
                         dy.numpy(), g.detach().numpy(), fc.detach().numpy(), stage_dtype=None)
    pairs = dict(dx=x, dw_g=w_g, dw_fc=w_fc, db_g=b_g, db_fc=b_fc)
    for name, t in pairs.items():
        ref = t.grad.numpy()
        got = np.asarray(out[name]).reshape(ref.shape)
        assert np.max(np.abs(got - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref))), name


def pin_linearity_in_dy():
    rng = _rng(8)
    M, K, N = 6, 4, 5
    x, w_g, w_fc = (rng.standard_normal(s) for s in ((M, K), (K, N), (K, N)))
    dy, g, fc = (rng.standard_normal((M, N)) for _ in range(3))
    a = osw.swiglu_bwd(x, w_g, w_fc, dy, g, fc, stage_dtype=None)
    b = osw.swiglu_bwd(x, w_g, w_fc, 2.0 * dy, g, fc, stage_dtype=None)
    c = osw.swiglu_bwd(x, w_g, w_fc, -dy, g, fc, stage_dtype=None)
    for k in a:
        assert np.array_equal(b[k], 2.0 * a[k]), k
        assert np.allclose(c[k], -a[k], rtol=0, atol=1e-15 * (1 + np.max(np.abs(a[k])))), k


def pin_sampled_matches_full():
    import torch
    rng = _rng(9)
    M, K, N = 40, 8, 16
    T = {n: torch.tensor(rng.standard_normal(s), dtype=torch.float64)
         for n, s in dict(x=(M, K), w_g=(K, N), w_fc=(K, N), dy=(M, N), g=(M, N), fc=(M, N)).items()}
    full = osw.swiglu_bwd(*(T[n].numpy() for n in ("x", "w_g", "w_fc", "dy", "g", "fc")))
    rows = np.array([0, 3, 17, 39])
    cols = np.array([1, 5, 15])
    s = osw.swiglu_bwd_sampled(T["x"], T["w_g"], T["w_fc"], T["dy"], T["g"], T["fc"], rows, cols)
    for k in ("dg", "dfc", "dx"):
        assert np.allclose(s[k], full[k][rows], rtol=1e-14, atol=1e-14), k
    for k in ("db_g", "db_fc", "dw_g", "dw_fc"):
        assert np.allclose(s[k], full[k][:, cols], rtol=1e-14, atol=1e-14), k


# --------------------------------------------------------------------------- SwishGrad

def _swish_local(x, beta):
    return x / (1.0 + np.exp(-beta * x))


def pin_swish_special_cases():
    rng = _rng(12)
    grad = rng.standard_normal(50)
    x = rng.standard_normal(50) * 4
    # beta = 0 or x = 0: sigma(0) = 1/2 and the bracket is 1, so grad_x = grad / 2 exactly
    assert np.array_equal(osh.swish_grad(grad, x, 0.0), grad / 2)
    assert np.array_equal(osh.swish_grad(grad, np.zeros(50), 1.702), grad / 2)
    # saturation: x -> +inf gives grad, x -> -inf gives 0
    assert np.allclose(osh.swish_grad(grad, np.full(50, 800.0), 1.0), grad, rtol=0, atol=0)
    assert np.all(osh.swish_grad(grad, np.full(50, -800.0), 1.0) == 0.0)
    # beta = 1: the SiLU derivative; grad = dy*fc, x = g reproduces dg of the SwiGLU b stage
    dy, g, fc = rng.standard_normal(50), rng.standard_normal(50) * 3, rng.standard_normal(50)
    dg, _, _, _ = osw.swiglu_bwd_b(dy[None], g[None], fc[None])
    assert np.allclose(osh.swish_grad(dy * fc, g, 1.0), dg[0], rtol=1e-15, atol=1e-300)


def pin_swish_alternative_form():
    # the page's first form: s'(x) = beta s(x) + sigma(beta x) (1 - beta s(x)), s(x) = x sigma(beta x)
    rng = _rng(13)
    x = rng.standard_normal(200) * 5
    for beta in (1.0, 1.702, 0.01, 1.1):
        b = float(np.float32(beta))
        sig = 1.0 / (1.0 + np.exp(-b * x))
        s = x * sig
        alt = b * s + sig * (1.0 - b * s)
        got = osh.swish_grad(np.ones_like(x), x, beta)
        assert np.allclose(got, alt, rtol=1e-13, atol=1e-15)


def pin_swish_fd():
    x = np.linspace(-20, 20, 161)
    for beta in (1.0, 1.702, 0.01):
        b = float(np.float32(beta))
        h = 1e-6 * np.maximum(1.0, np.abs(x))
        fd = (_swish_local(x + h, b) - _swish_local(x - h, b)) / (2 * h)
        got = osh.swish_grad(np.ones_like(x), x, beta)
        assert np.max(np.abs(got - fd)) < 1e-7, beta


def pin_swish_cann_sample():
    import sympy as sp
    with open(os.path.join(GOLDEN, "swishgrad_cann_sample.json")) as f:
        case = json.load(f)
    beta32 = float(np.float32(case["beta"]))
    xs, bs = sp.symbols("x b")
    d = sp.diff(xs / (1 + sp.exp(-bs * xs)), xs)
    ref = np.array([float(d.subs({xs: v, bs: sp.Float(beta32, 40)}).evalf(40)) for v in case["x"]])
    ref = ref * np.array(case["grad"], dtype=np.float64)
    got = osh.swish_grad(np.array(case["grad"], np.float64), np.array(case["x"], np.float64),
                         case["beta"])
    assert np.all(np.abs(got - ref) <= 1e-14 * np.abs(ref)), (got, ref)
    # the same six values once rounded to fp32, the sample's dtype
    assert np.array_equal(onum.round_to_dtype(got, "f32"), ref.astype(np.float32).astype(np.float64))


# --------------------------------------------------------------------------- bf16 codec

def pin_bf16_rounding():
    import torch
    rng = _rng(17)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, 3.0e38, -3.0e38, 1e-40, -1e-41])]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = onum.f64_to_bf16_bits(v.astype(np.float64))
    assert np.array_equal(got, want)
    # ties go to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert onum.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert onum.f64_to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
    # direct rounding from fp64: just above the halfway point must round up,
    # although rounding to fp32 first would land exactly on the tie
    assert onum.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    # widening is exact and inverts narrowing on every bf16 pattern
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = onum.bf16_bits_to_f64(allbits)
    finite = np.isfinite(vals)
    rt = onum.f64_to_bf16_bits(vals[finite])
    # -0.0 and +0.0 both survive (sign kept by frexp/ldexp)
    assert np.array_equal(rt, allbits[finite])


# --------------------------------------------------------------------------- forward

def pin_forward_bruteforce():
    """g, fc by explicit loops with the bias, y = g * sigma(g) * fc per element
    with the textbook sigmoid 1 / (1 + e^-g) (finite for these inputs)."""
    rng = _rng(41)
    M, K, N = 3, 4, 5
    x, w_g, w_fc = rng.standard_normal((M, K)), rng.standard_normal((K, N)), rng.standard_normal((K, N))
    b_g, b_fc = rng.standard_normal(N), rng.standard_normal(N)
    g, fc, y = osw.swiglu_fwd(x, w_g, w_fc, b_g, b_fc)
    for i in range(M):
        for j in range(N):
            gij = b_g[j] + sum(x[i, k] * w_g[k, j] for k in range(K))
            fij = b_fc[j] + sum(x[i, k] * w_fc[k, j] for k in range(K))
            yij = gij / (1.0 + math.exp(-gij)) * fij
            assert abs(g[i, j] - gij) < 1e-13 and abs(fc[i, j] - fij) < 1e-13
            assert abs(y[i, j] - yij) < 1e-13 * max(1.0, abs(yij))


def pin_forward_torch():
    import torch
    rng = _rng(43)
    M, K, N = 9, 7, 11
    x, w_g, w_fc = rng.standard_normal((M, K)), rng.standard_normal((K, N)), rng.standard_normal((K, N))
    b_g, b_fc = rng.standard_normal(N), rng.standard_normal(N)
    t = lambda a: torch.tensor(a, dtype=torch.float64)  # noqa: E731
    ref = torch.nn.functional.silu(t(x) @ t(w_g) + t(b_g)) * (t(x) @ t(w_fc) + t(b_fc))
    _, _, y = osw.swiglu_fwd(x, w_g, w_fc, b_g, b_fc)
    assert np.max(np.abs(y - ref.numpy())) < 1e-12


def pin_forward_closed_forms():
    """With K = 1 and x = 1 the gate takes chosen values: sigma(0) = 1/2,
    sigma(ln 3) = 3/4, sigma(-ln 3) = 1/4, so y = g * sigma(g) * fc is known exactly."""
    l3 = math.log(3.0)
    x = np.array([[1.0]])
    w_g = np.array([[0.0, l3, -l3]])
    w_fc = np.array([[2.0, 2.0, 2.0]])
    g, fc, y = osw.swiglu_fwd(x, w_g, w_fc, None, np.array([0.0, 1.0, -1.0]))
    assert np.allclose(g, [[0.0, l3, -l3]], rtol=0, atol=1e-15)
    assert np.allclose(fc, [[2.0, 3.0, 1.0]], rtol=0, atol=1e-15)
    assert np.allclose(y, [[0.0, l3 * 0.75 * 3.0, -l3 * 0.25 * 1.0]], rtol=1e-15, atol=1e-15)


# --------------------------------------------------------------------------- sibling activations

def _gelu_local(z):
    return z * 0.5 * (1.0 + math.erf(z / math.sqrt(2.0)))


def _hardswish_local(z):
    return z * min(max(z + 3.0, 0.0), 6.0) / 6.0


def pin_gelu_grad_fd():
    z = np.concatenate([np.linspace(-8, 8, 161), _rng(51).standard_normal(200) * 3])
    h = 1e-6
    fd = np.array([(_gelu_local(v + h) - _gelu_local(v - h)) / (2 * h) for v in z])
    assert np.max(np.abs(oact.gelu_grad(np.ones_like(z), z) - fd)) < 1e-8


def pin_gelu_grad_torch_and_special_values():
    import torch
    z = np.concatenate([np.linspace(-10, 10, 201), _rng(53).standard_normal(300) * 4])
    t = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(t, approximate="none").sum().backward()
    assert np.max(np.abs(oact.gelu_grad(np.ones_like(z), z) - t.grad.numpy())) < 1e-14
    g = oact.gelu_grad(np.array([2.0, 2.0, 2.0]), np.array([0.0, 40.0, -40.0]))
    assert g[0] == 1.0 and g[1] == 2.0 and g[2] == 0.0  # GELU'(0) = 1/2; saturation


def pin_hardswish_grad():
    import torch
    z = np.concatenate([np.linspace(-5, 5, 1001), [-3.0, 3.0, -4.0, 4.0, 0.0], _rng(55).standard_normal(300) * 3])
    t = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.hardswish(t).sum().backward()
    got = oact.hardswish_grad(np.ones_like(z), z)
    assert np.max(np.abs(got - t.grad.numpy())) < 1e-15
    # finite differences away from the kinks; slope 1/3 in the middle; flat outside
    h = 1e-6
    w = z[(np.abs(z + 3) > 1e-3) & (np.abs(z - 3) > 1e-3)]
    fd = np.array([(_hardswish_local(v + h) - _hardswish_local(v - h)) / (2 * h) for v in w])
    assert np.max(np.abs(oact.hardswish_grad(np.ones_like(w), w) - fd)) < 1e-8
    v = oact.hardswish_grad(np.ones(5), np.array([-4.0, -3.0, 0.0, 3.0, 4.0]))
    assert list(v) == [0.0, 0.0, 0.5, 1.0, 1.0]


# --------------------------------------------------------------------------- GroupNorm backward

def _gn_inputs(N, C, S, G, seed):
    """x with a different mean and spread per (sample, group), dy, gamma, beta."""
    r = _rng(seed)
    loc = r.uniform(-2, 2, (N, G, 1, 1))
    sc = r.uniform(0.5, 2.0, (N, G, 1, 1))
    x = (loc + sc * r.standard_normal((N, G, C // G, S))).reshape(N, C, S)
    return x, r.standard_normal((N, C, S)), 1.0 + 0.5 * r.standard_normal(C), r.standard_normal(C)


def _gn_loss_local(x, gamma, beta, dy, G, eps):
    """sum(dy * GroupNorm(x)), the forward written out group by group with explicit loops."""
    N, C, S = x.shape
    cg = C // G
    total = 0.0
    for n in range(N):
        for g in range(G):
            vals = [x[n, c, s] for c in range(g * cg, (g + 1) * cg) for s in range(S)]
            mu = sum(vals) / len(vals)
            var = sum((v - mu) ** 2 for v in vals) / len(vals)
            inv = 1.0 / math.sqrt(var + eps)
            for c in range(g * cg, (g + 1) * cg):
                for s in range(S):
                    total += dy[n, c, s] * (gamma[c] * (x[n, c, s] - mu) * inv + beta[c])
    return total


def pin_group_norm_fd():
    N, C, S, G, eps = 2, 6, 5, 3, 1e-3
    x, dy, gamma, beta = _gn_inputs(N, C, S, G, 60)
    dx, dgamma, dbeta = ogn.group_norm_bwd(dy, x, gamma, G, eps)
    h = 1e-5

    def fd(arr, idx):
        a0 = arr[idx]
        arr[idx] = a0 + h
        lp = _gn_loss_local(x, gamma, beta, dy, G, eps)
        arr[idx] = a0 - h
        lm = _gn_loss_local(x, gamma, beta, dy, G, eps)
        arr[idx] = a0
        return (lp - lm) / (2 * h)

    fdx = np.array([fd(x, i) for i in np.ndindex(x.shape)]).reshape(x.shape)
    fdg = np.array([fd(gamma, (c,)) for c in range(C)])
    fdb = np.array([fd(beta, (c,)) for c in range(C)])
    assert np.max(np.abs(dx - fdx)) < 1e-7 * max(1.0, np.max(np.abs(fdx)))
    assert np.max(np.abs(dgamma - fdg)) < 1e-7 * max(1.0, np.max(np.abs(fdg)))
    assert np.max(np.abs(dbeta - fdb)) < 1e-7 * max(1.0, np.max(np.abs(fdb)))


def pin_group_norm_torch():
    import torch
    for (N, C, S, G, eps) in [(3, 8, 7, 4, 1e-5), (2, 6, 9, 1, 1e-5), (2, 6, 4, 6, 1e-2)]:
        x, dy, gamma, beta = _gn_inputs(N, C, S, G, 61 + G)
        xt = torch.tensor(x, requires_grad=True)
        gt = torch.tensor(gamma, requires_grad=True)
        bt = torch.tensor(beta, requires_grad=True)
        torch.nn.functional.group_norm(xt, G, gt, bt, eps).backward(torch.tensor(dy))
        dx, dgamma, dbeta = ogn.group_norm_bwd(dy, x, gamma, G, eps)
        assert np.max(np.abs(dx - xt.grad.numpy())) < 1e-12 * max(1.0, np.max(np.abs(dx)))
        assert np.max(np.abs(dgamma - gt.grad.numpy())) < 1e-11
        assert np.max(np.abs(dbeta - bt.grad.numpy())) < 1e-11


def pin_group_norm_invariants():
    N, C, S, G = 3, 8, 11, 2
    x, dy, gamma, _ = _gn_inputs(N, C, S, G, 62)
    # with eps = 0 the output ignores a shift or a scaling of x within a group, so dx is
    # orthogonal to the constants and to (x - mu) in every group
    dx, _, _ = ogn.group_norm_bwd(dy, x, gamma, G, 0.0)
    xg = x.reshape(N, G, -1)
    dg = dx.reshape(N, G, -1)
    mu = np.array([[np.mean(xg[n, g]) for g in range(G)] for n in range(N)])
    assert np.max(np.abs(dg.sum(axis=2))) < 1e-11
    assert np.max(np.abs((dg * (xg - mu[:, :, None])).sum(axis=2))) < 1e-10
    # statistics against plain per-slice numpy; dbeta and dgamma against loops
    mu_o, var_o, rstd_o = ogn.group_norm_stats(x, G, 1e-5)
    assert np.allclose(mu_o, mu, rtol=0, atol=1e-14)
    var = np.array([[np.var(xg[n, g]) for g in range(G)] for n in range(N)])
    assert np.allclose(var_o, var, rtol=1e-14, atol=0)
    _, dgamma, dbeta = ogn.group_norm_bwd(dy, x, gamma, G, 1e-5)
    cg = C // G
    for c in range(C):
        g = c // cg
        b = sum(dy[n, c, s] for n in range(N) for s in range(S))
        gm = sum(dy[n, c, s] * (x[n, c, s] - mu[n, g]) / math.sqrt(var[n, g] + 1e-5)
                 for n in range(N) for s in range(S))
        assert abs(dbeta[c] - b) < 1e-12 and abs(dgamma[c] - gm) < 1e-11
    # gamma None is gamma = 1
    a = ogn.group_norm_bwd(dy, x, None, G, 1e-5)
    b = ogn.group_norm_bwd(dy, x, np.ones(C), G, 1e-5)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    # one element per group (C = G, HxW = 1): the output is beta whatever x is, so dx = 0, dgamma = 0
    x1 = _rng(63).standard_normal((4, 5, 1))
    d1, g1, b1 = ogn.group_norm_bwd(_rng(64).standard_normal((4, 5, 1)), x1, np.full(5, 2.0), 5, 1e-5)
    assert np.max(np.abs(d1)) < 1e-12 and np.max(np.abs(g1)) == 0.0


ALL_PINS = [
    pin_sigmoid_closed_forms, pin_sigmoid_matches_scipy, pin_sigmoid_derivative,
    pin_silu_grad_fd, pin_silu_grad_symbolic, pin_b_stage_symbolic, pin_b_stage_fd,
    pin_db_is_column_sum, pin_gemm_bruteforce, pin_full_chain_fd, pin_torch_autograd,
    pin_linearity_in_dy, pin_sampled_matches_full, pin_swish_special_cases,
    pin_swish_alternative_form, pin_swish_fd, pin_swish_cann_sample, pin_bf16_rounding,
    pin_forward_bruteforce, pin_forward_torch, pin_forward_closed_forms,
    pin_gelu_grad_fd, pin_gelu_grad_torch_and_special_values, pin_hardswish_grad,
    pin_group_norm_fd, pin_group_norm_torch, pin_group_norm_invariants,
]
