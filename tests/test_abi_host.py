"""The C-ABI library on the host: it loads, exports every function that
include/*.h declares, and rejects bad arguments before any device work.

These calls pass fake, never-dereferenced addresses: every case returns from
the argument checks before any CUDA call, so no GPU is needed.
"""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def swg():
    import swiglu_ffn_backward_gb300 as m
    return m


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("swiglu_bwd", "swiglu_bwd_b", "swiglu_bwd_w", "swiglu_bwd_x", "swish_grad",
              "swiglu_bwd_workspace_size", "swg_status_string", "swg_check"):
        assert n in names


def test_library_exports_every_declared_symbol(swg):
    lib = ctypes.CDLL(swg.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(swg.EXPORTS) <= _declared_functions()


def test_status_strings(swg):
    from swiglu_ffn_backward_gb300 import _binding as b
    for code in range(7):
        s = b.status_string(code)
        assert s.startswith("SWG_")
    assert "unknown" in b.status_string(99)


FAKE = 0x7f0000000000  # 16-byte aligned, never dereferenced


def _lib(swg):
    from swiglu_ffn_backward_gb300 import _binding as b
    return b.lib, b


def test_null_pointers(swg):
    lib, b = _lib(swg)
    assert lib.swish_grad(None, FAKE, None, FAKE, 10, b.SWG_F32, None) == b.SWG_ERR_NULLPTR
    assert lib.swiglu_bwd_b(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 8, None, 0, None) == b.SWG_ERR_NULLPTR
    assert lib.swiglu_bwd_w(FAKE, FAKE, None, FAKE, FAKE, 4, 8, 8, None, 0, None) == b.SWG_ERR_NULLPTR
    assert lib.swiglu_bwd_x(FAKE, FAKE, FAKE, FAKE, None, 4, 8, 8, None) == b.SWG_ERR_NULLPTR
    # dg given without dfc
    args = [FAKE + i * 0x1000000 for i in range(13)]
    args[7] = None
    assert lib.swiglu_bwd(*args, 4, 8, 8, 0, None, 0, None) == b.SWG_ERR_NULLPTR


def test_invalid_sizes_and_dtypes(swg):
    lib, b = _lib(swg)
    assert lib.swish_grad(FAKE, FAKE + 4096, None, FAKE + 8192, -1, b.SWG_F32, None) == b.SWG_ERR_PARAM_INVALID
    assert lib.swish_grad(FAKE, FAKE + 4096, None, FAKE + 8192, 10, 7, None) == b.SWG_ERR_PARAM_INVALID
    assert lib.swiglu_bwd_x(FAKE, FAKE + 2**24, FAKE + 2**25, FAKE + 2**26, FAKE + 2**27, -1, 8, 8,
                            None) == b.SWG_ERR_PARAM_INVALID
    base = [FAKE + i * 2**26 for i in range(13)]
    assert lib.swiglu_bwd(*base, 4, 8, 8, 0x40, None, 0, None) == b.SWG_ERR_PARAM_INVALID  # unknown flag


def test_unsupported_shapes_and_alignment(swg):
    lib, b = _lib(swg)
    p = [FAKE + i * 2**26 for i in range(7)]
    # N not a multiple of 8
    assert lib.swiglu_bwd_b(*p, 16, 12, None, 0, None) == b.SWG_ERR_UNSUPPORTED
    # K not a multiple of 8
    assert lib.swiglu_bwd_x(p[0], p[1], p[2], p[3], p[4], 16, 12, 16, None) == b.SWG_ERR_UNSUPPORTED
    # misaligned pointer
    q = list(p)
    q[2] += 2
    assert lib.swiglu_bwd_b(*q, 16, 16, None, 0, None) == b.SWG_ERR_UNSUPPORTED
    # fp32 swish_grad pointer not 4-byte aligned
    assert lib.swish_grad(FAKE + 2, FAKE + 4096, None, FAKE + 8192, 10, b.SWG_F32, None) == b.SWG_ERR_UNSUPPORTED
    # M beyond 32-bit TMA coordinates
    assert lib.swiglu_bwd_x(p[0], p[1], p[2], p[3], p[4], 2**31, 8, 8, None) == b.SWG_ERR_UNSUPPORTED


def test_overlapping_buffers(swg):
    lib, b = _lib(swg)
    M, N = 64, 64
    mn = M * N * 2
    dy, g, fc = FAKE, FAKE + mn, FAKE + 2 * mn
    # dg overlaps fc
    assert lib.swiglu_bwd_b(dy, g, fc, fc + 16, FAKE + 8 * mn, FAKE + 10 * mn, FAKE + 11 * mn, M, N,
                            None, 0, None) == b.SWG_ERR_PARAM_INVALID
    # grad_x partially overlapping grad is rejected (exact aliasing is allowed)
    assert lib.swish_grad(FAKE, FAKE + 4096, None, FAKE + 16, 100, b.SWG_F32, None) == b.SWG_ERR_PARAM_INVALID


def test_workspace_queries(swg):
    assert swg.swiglu_bwd_b_workspace_size(0, 1024) == 0
    assert swg.swiglu_bwd_b_workspace_size(220000, 1024) > 0
    assert swg.swiglu_bwd_b_workspace_size(220000, 1024) % 16 == 0
    # the unfused whole backward needs room for dg, dfc unless the caller passes them
    M, K, N = 220000, 512, 1024
    assert swg.swiglu_bwd_workspace_size(M, K, N, 0) >= 4 * M * N
    assert swg.swiglu_bwd_workspace_size(M, K, N, 0x100) < 4 * M * N


def test_python_binding_requires_cuda_tensors(swg):
    import torch
    t = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        swg.swiglu_bwd_b(t, t, t)
    with pytest.raises(TypeError):
        swg.swish_grad(t, t, 1.0)


def test_forward_argument_checks(swg):
    lib, b = _lib(swg)
    p = [FAKE + i * 2**26 for i in range(8)]  # x, w_g, w_fc, b_g, b_fc, g, fc, y
    assert lib.swiglu_fwd(None, *p[1:], 16, 8, 8, None) == b.SWG_ERR_NULLPTR
    assert lib.swiglu_fwd(*p[:7], None, 16, 8, 8, None) == b.SWG_ERR_NULLPTR
    assert lib.swiglu_fwd(*p, -1, 8, 8, None) == b.SWG_ERR_PARAM_INVALID
    assert lib.swiglu_fwd(*p, 16, 12, 8, None) == b.SWG_ERR_UNSUPPORTED   # K not a multiple of 8
    assert lib.swiglu_fwd(*p, 16, 0, 8, None) == b.SWG_ERR_UNSUPPORTED    # no reduction to run
    q = list(p)
    q[3] += 2  # misaligned bias
    assert lib.swiglu_fwd(*q, 16, 8, 8, None) == b.SWG_ERR_UNSUPPORTED
    q = list(p)
    q[7] = q[6] + 16  # y overlaps fc
    assert lib.swiglu_fwd(*q, 16, 8, 8, None) == b.SWG_ERR_PARAM_INVALID
    # empty M: nothing to do, even with NULL buffers
    assert lib.swiglu_fwd(None, p[1], p[2], None, None, None, None, None, 0, 8, 8, None) == b.SWG_OK


def test_accumulate_flag_is_accepted_and_empty_M_needs_no_device(swg):
    lib, b = _lib(swg)
    base = [FAKE + i * 2**26 for i in range(13)]
    base[0] = base[3] = base[4] = base[5] = base[8] = None  # x, dy, g, fc, dx are empty at M = 0
    base[6] = base[7] = None  # no dg, dfc
    # M = 0 with SWG_ACCUMULATE returns before touching the device (no GPU here)
    assert lib.swiglu_bwd(*base, 0, 8, 8, b.SWG_ACCUMULATE, None, 0, None) == b.SWG_OK
    assert lib.swiglu_bwd(*base, 0, 8, 8, b.SWG_ACCUMULATE | b.SWG_FUSED, None, 0, None) == b.SWG_OK


def test_forward_binding_checks_shapes(swg):
    import torch
    t = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        swg.swiglu_fwd(t, t, t)


def test_act_grad_argument_checks(swg):
    lib, b = _lib(swg)
    assert lib.act_grad(FAKE, FAKE + 4096, 7, FAKE + 8192, 10, b.SWG_F32, None) == b.SWG_ERR_PARAM_INVALID
    assert lib.act_grad(FAKE, None, 1, FAKE + 8192, 10, b.SWG_F32, None) == b.SWG_ERR_NULLPTR
    assert lib.act_grad(FAKE, FAKE + 4096, 1, FAKE + 16, 100, b.SWG_F32, None) == b.SWG_ERR_PARAM_INVALID
    assert lib.act_grad(None, None, 2, None, 0, b.SWG_BF16, None) == b.SWG_OK  # empty


def test_group_norm_argument_checks(swg):
    lib, b = _lib(swg)
    gn = lib.group_norm_bwd
    A = [FAKE + i * 0x1000000 for i in range(6)]  # dy, x, gamma, dx, dgamma, dbeta
    ws_ok = lib.group_norm_bwd_workspace_size(2, 8, 12, 4)
    assert ws_ok > 0 and lib.group_norm_bwd_workspace_size(2, 8, 12, 3) == 0
    assert lib.group_norm_bwd_workspace_size(0, 8, 12, 4) == 0
    # G < 1, C not a multiple of G, negative sizes, NaN / negative eps, bad dtype
    assert gn(*A, 2, 8, 12, 0, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    assert gn(*A, 2, 8, 12, 3, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    assert gn(*A, -1, 8, 12, 4, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    assert gn(*A, 2, 8, 12, 4, float("nan"), b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    assert gn(*A, 2, 8, 12, 4, -1.0, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    assert gn(*A, 2, 8, 12, 4, 1e-5, 9, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    # too many (sample, group) pairs for the grid; an element count past 2^60
    assert gn(*A, 1 << 19, 1 << 9, 1, 1 << 9, 1e-5, b.SWG_F32, FAKE, 1 << 40, None) == b.SWG_ERR_UNSUPPORTED
    assert gn(*A, 1 << 20, 1 << 20, 1 << 21, 1, 1e-5, b.SWG_F32, FAKE, 1 << 40, None) == b.SWG_ERR_UNSUPPORTED
    # NULL x, dy or dx for a non-empty tensor
    for i in (0, 1, 3):
        args = list(A)
        args[i] = None
        assert gn(*args, 2, 8, 12, 4, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_NULLPTR
    # pointers not aligned to the element size
    args = list(A)
    args[1] = FAKE + 2
    assert gn(*args, 2, 8, 12, 4, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_UNSUPPORTED
    # dx overlapping x; dgamma overlapping gamma
    args = list(A)
    args[3] = A[1] + 64
    assert gn(*args, 2, 8, 12, 4, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    args = list(A)
    args[4] = A[2]
    assert gn(*args, 2, 8, 12, 4, 1e-5, b.SWG_F32, FAKE, ws_ok, None) == b.SWG_ERR_PARAM_INVALID
    # dgamma / dbeta wanted: workspace missing, short or misaligned
    assert gn(*A, 2, 8, 12, 4, 1e-5, b.SWG_F32, None, 0, None) == b.SWG_ERR_WORKSPACE
    assert gn(*A, 2, 8, 12, 4, 1e-5, b.SWG_F32, FAKE, ws_ok - 1, None) == b.SWG_ERR_WORKSPACE
    assert gn(*A, 2, 8, 12, 4, 1e-5, b.SWG_F32, FAKE + 8, ws_ok, None) == b.SWG_ERR_WORKSPACE
    # empty without parameter gradients: nothing to do, no device needed, NULL data pointers accepted
    assert gn(None, None, None, None, None, None, 0, 8, 12, 4, 1e-5, b.SWG_BF16, None, 0, None) == b.SWG_OK
    assert gn(None, None, None, None, None, None, 2, 8, 0, 4, 1e-5, b.SWG_F16, None, 0, None) == b.SWG_OK


def test_host_path_argument_checks(swg):
    lib, b = _lib(swg)
    A = [FAKE + i * 0x1000000 for i in range(11)]  # x, w_g, w_fc, dy, g, fc, dx, dw_g, dw_fc, db_g, db_fc
    assert lib.swiglu_bwd_host_workspace_size(220000, 512, 1024) > 0
    assert lib.swiglu_bwd_host_workspace_size(-1, 512, 1024) == 0
    # K, N not multiples of 8; negative M
    assert lib.swiglu_bwd_host(*A, 4, 12, 16, FAKE, 1 << 30, None) == b.SWG_ERR_UNSUPPORTED
    assert lib.swiglu_bwd_host(*A, -1, 8, 16, FAKE, 1 << 30, None) == b.SWG_ERR_PARAM_INVALID
    # NULL weights, outputs or (M > 0) activations
    for i in (1, 6, 7, 10, 0, 3):
        args = list(A)
        args[i] = None
        assert lib.swiglu_bwd_host(*args, 4, 8, 16, FAKE, 1 << 30, None) == b.SWG_ERR_NULLPTR, i
    # dx overlapping dy
    args = list(A)
    args[6] = A[3] + 16
    assert lib.swiglu_bwd_host(*args, 4, 8, 16, FAKE, 1 << 30, None) == b.SWG_ERR_PARAM_INVALID


def _al256(v):
    return (v + 255) & ~255


def _fw_splits(M, K, N, sms):
    nkb = (M + 63) // 64
    tiles = ((N + 63) // 64) * ((K + 511) // 512)
    s = max(1, sms // tiles)
    s = min(s, max(1, nkb // 8), 64)
    kb_per = (nkb + s - 1) // s if nkb > 0 else 0
    return (nkb + kb_per - 1) // kb_per if kb_per > 0 else 1


def _fw_ws(M, K, N, sms):
    s = _fw_splits(M, K, N, sms)
    return _al256(s * 2 * K * N * 4 if s > 1 else 0) + _al256(s * 2 * N * 4)


@pytest.mark.parametrize("M", [0, 256, 40000, 65535, 65536, 70001, 220000, 3_000_000])
def test_host_path_workspace_follows_the_chunk_plan(swg, M):
    # without a device the library plans for 148 SMs; the layout: W | 2 input sets | 2 dx sets |
    # outputs | partials of every chunk (or the fused w stage's own workspace for one chunk)
    K, N, sms = 512, 1024, 148
    chunks = min(M // 32768, 256) if M >= 65536 else (1 if M > 0 else 0)
    # equal chunks of a 64-row multiple, then the shortest last chunk the partials path allows
    rows = (M - 16384) // (chunks - 1) // 64 * 64 if chunks > 1 else (M + 63) // 64 * 64
    if chunks > 1:
        last = M - (chunks - 1) * rows
        assert 16384 <= last <= min(rows, 16384 + 64 * (chunks - 1))  # every chunk splits over M
    total = _al256(2 * K * N * 2) + 2 * _al256(rows * (K + 3 * N) * 2) + 2 * _al256(rows * K * 2)
    total += _al256((2 * K * N + 2 * N) * 2)
    if chunks > 1:
        st = sum(_fw_splits(min(rows, M - c * rows), K, N, sms) for c in range(chunks))
        total += _al256(st * 2 * K * N * 4) + _al256(st * 2 * N * 4)
    elif chunks == 1:
        total += _al256(_fw_ws(M, K, N, sms))
    assert swg.swiglu_bwd_host_workspace_size(M, K, N) == total


def test_host_path_binding_checks_buffers(swg):
    import torch
    bf = dict(dtype=torch.bfloat16)
    M, K, N = 4, 8, 16
    ins = dict(x=torch.zeros(M, K, **bf), w_g=torch.zeros(K, N, **bf), w_fc=torch.zeros(K, N, **bf),
               dy=torch.zeros(M, N, **bf), g=torch.zeros(M, N, **bf), fc=torch.zeros(M, N, **bf))
    with pytest.raises(ValueError):  # a short output would be overrun by the copies
        swg.swiglu_bwd_host(**ins, out={"dx": torch.zeros(M, K - 1, **bf)})
    with pytest.raises(ValueError):  # dy with the wrong row count
        swg.swiglu_bwd_host(**dict(ins, dy=torch.zeros(M + 1, N, **bf)))
    with pytest.raises(TypeError):   # fp32 inputs
        swg.swiglu_bwd_host(**dict(ins, x=torch.zeros(M, K)))


def test_auto_flag_resolves_like_the_measured_choice(swg):
    """SWG_AUTO takes the fused chain for K <= 512 and M >= 32768, else the unfused one;
    the workspace query resolves it the same way."""
    from swiglu_ffn_backward_gb300 import _binding as b
    q = b.lib.swiglu_bwd_workspace_size
    for M, K, N, fused in ((220000, 512, 1024, True), (65537, 512, 1024, True), (4097, 512, 1024, False),
                           (16384, 4096, 14336, False), (32767, 512, 1024, False)):
        want = q(M, K, N, b.SWG_FUSED if fused else b.SWG_UNFUSED)
        assert q(M, K, N, b.SWG_AUTO) == want, (M, K, N)
        assert q(M, K, N, b.SWG_AUTO | b.SWG_ACCUMULATE) == q(M, K, N, (b.SWG_FUSED if fused else 0)
                                                                | b.SWG_ACCUMULATE)


def test_kernel_count_query(swg):
    # without a device the library plans for 148 SMs: the w stage takes 144 CTAs at the pages'
    # shape, and the four free SMs could not finish the x stage's extra tiles inside it, so the
    # fused call is x stage + w stage + one launch for its two reductions; the unfused one adds
    # the b stage's db reduction and the w GEMM's split reduction to its three stages
    assert swg.swiglu_bwd_kernel_count(220000, 512, 1024, swg.SWG_FUSED) == 3
    assert swg.swiglu_bwd_kernel_count(220000, 512, 1024, swg.SWG_UNFUSED) == 5
    assert swg.swiglu_bwd_kernel_count(220000, 512, 1024, swg.SWG_AUTO) == 3
    assert swg.swiglu_bwd_kernel_count(0, 512, 1024, swg.SWG_FUSED) == 0  # memsets only
    assert swg.swiglu_bwd_kernel_count(100, 0, 1024, swg.SWG_FUSED) == 0
    assert swg.swiglu_bwd_kernel_count(100, 512, 1020, swg.SWG_FUSED) == 0  # N not a multiple of 8
    assert swg.swiglu_bwd_kernel_count(100, 512, 1024, 0x80) == 0  # unknown flag
