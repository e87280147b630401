"""ctypes binding of include/swiglu_bwd.h: argument marshalling only.

Every step of the backward runs in the library's sm_103a kernels. torch is
used for device memory (outputs and workspace are allocated with torch.empty
when the caller passes none) and for the current CUDA stream. If the shared
library is missing the import of this module raises: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libswiglu_bwd.so")

# status codes (swg_status)
SWG_OK = 0
SWG_ERR_NULLPTR = 1
SWG_ERR_PARAM_INVALID = 2
SWG_ERR_UNSUPPORTED = 3
SWG_ERR_WORKSPACE = 4
SWG_ERR_CUDA = 5
SWG_ERR_TIMEOUT = 6

# dtypes (swg_dtype)
SWG_F32, SWG_F16, SWG_BF16 = 0, 1, 2
_DTYPE = {torch.float32: SWG_F32, torch.float16: SWG_F16, torch.bfloat16: SWG_BF16}

# flags
SWG_UNFUSED = 0
SWG_FUSED = 1
SWG_ACCUMULATE = 2
SWG_AUTO = 4
SWG_WS_DG_GIVEN = 0x100

EXPORTS = (
    "swg_status_string", "swg_check",
    "swiglu_bwd_b_workspace_size", "swiglu_bwd_b",
    "swiglu_bwd_w_workspace_size", "swiglu_bwd_w",
    "swiglu_bwd_x",
    "swiglu_bwd_workspace_size", "swiglu_bwd", "swiglu_bwd_kernel_count",
    "swish_grad",
    "swiglu_bwd_b_noalloc",
    "swiglu_bwd_x_fused",
    "swiglu_bwd_w_fused_workspace_size", "swiglu_bwd_w_fused",
    "swiglu_fwd",
    "act_grad",
    "group_norm_bwd_workspace_size", "group_norm_bwd",
    "swiglu_bwd_host_workspace_size", "swiglu_bwd_host",
    "swg_inject_stall",
)


class SwgError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python swiglu_ffn_backward_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, SZ, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint
    st = ctypes.c_int
    lib.swg_status_string.argtypes = [st]
    lib.swg_status_string.restype = ctypes.c_char_p
    lib.swg_check.argtypes = [P]
    lib.swg_check.restype = st
    lib.swg_inject_stall.argtypes = [ctypes.c_int, I64, I64]
    lib.swg_inject_stall.restype = st
    lib.swiglu_bwd_b_workspace_size.argtypes = [I64, I64]
    lib.swiglu_bwd_b_workspace_size.restype = SZ
    lib.swiglu_bwd_b.argtypes = [P, P, P, P, P, P, P, I64, I64, P, SZ, P]
    lib.swiglu_bwd_b.restype = st
    lib.swiglu_bwd_w_workspace_size.argtypes = [I64, I64, I64]
    lib.swiglu_bwd_w_workspace_size.restype = SZ
    lib.swiglu_bwd_w.argtypes = [P, P, P, P, P, I64, I64, I64, P, SZ, P]
    lib.swiglu_bwd_w.restype = st
    lib.swiglu_bwd_x.argtypes = [P, P, P, P, P, I64, I64, I64, P]
    lib.swiglu_bwd_x.restype = st
    lib.swiglu_fwd.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I64, P]
    lib.swiglu_fwd.restype = st
    lib.act_grad.argtypes = [P, P, ctypes.c_int, P, I64, ctypes.c_int, P]
    lib.swiglu_bwd_host_workspace_size.restype = SZ
    lib.swiglu_bwd_host_workspace_size.argtypes = [I64, I64, I64]
    lib.swiglu_bwd_host.restype = st
    lib.swiglu_bwd_host.argtypes = [P] * 11 + [I64, I64, I64, P, SZ, P]
    lib.group_norm_bwd_workspace_size.restype = SZ
    lib.group_norm_bwd_workspace_size.argtypes = [I64, I64, I64, I64]
    lib.group_norm_bwd.restype = st
    lib.group_norm_bwd.argtypes = [P] * 6 + [I64, I64, I64, I64, ctypes.c_float, ctypes.c_int, P, SZ, P]
    lib.act_grad.restype = st
    lib.swiglu_bwd_workspace_size.argtypes = [I64, I64, I64, U]
    lib.swiglu_bwd_workspace_size.restype = SZ
    lib.swiglu_bwd_kernel_count.argtypes = [I64, I64, I64, U]
    lib.swiglu_bwd_kernel_count.restype = ctypes.c_int
    lib.swiglu_bwd.argtypes = [P] * 13 + [I64, I64, I64, U, P, SZ, P]
    lib.swiglu_bwd.restype = st
    lib.swish_grad.argtypes = [P, P, ctypes.POINTER(ctypes.c_float), P, I64, ctypes.c_int, P]
    lib.swish_grad.restype = st
    lib.swiglu_bwd_b_noalloc.argtypes = [P, P, P, P, P, P, P, I64, I64, P]
    lib.swiglu_bwd_b_noalloc.restype = st
    lib.swiglu_bwd_x_fused.argtypes = [P] * 8 + [I64, I64, I64, P]
    lib.swiglu_bwd_x_fused.restype = st
    lib.swiglu_bwd_w_fused_workspace_size.argtypes = [I64, I64, I64]
    lib.swiglu_bwd_w_fused_workspace_size.restype = SZ
    lib.swiglu_bwd_w_fused.argtypes = [P] * 8 + [I64, I64, I64, P, SZ, P]
    lib.swiglu_bwd_w_fused.restype = st
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.swg_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != SWG_OK:
        raise SwgError(status, f"{what}: {status_string(status)}")


def _stream(stream=None, device=None) -> int:
    """The raw handle of `stream`, or of the current stream of `device` when
    stream is None. A torch stream of another device is refused: the kernels
    would run on the wrong GPU."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if hasattr(stream, "cuda_stream"):
        if device is not None and getattr(stream, "device", None) is not None and \
                torch.device(stream.device) != torch.device(device):
            raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
        return stream.cuda_stream
    return int(stream)


def _device_of(*tensors) -> torch.device:
    """The one CUDA device that every given tensor (None skipped) lives on.
    The library launches on the current device, so tensors spread over two
    GPUs, or on a GPU other than the current one without the switch below,
    would be read through the wrong device's address space."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"all tensors must be on one device: got {dev} and {t.device}")
    return dev


def _call(dev, fn, *args):
    """Run one C-ABI call with `dev` as the current device (and so the device
    the library resolves its launch configuration and status word on)."""
    with torch.cuda.device(dev):
        return fn(*args)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dev_bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bf16, got {t.dtype}")
    return t.contiguous()


def _workspace(nbytes: int, device, given):
    if given is not None:
        return given
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _out(t, shape, dtype, device, name="output"):
    """An output buffer: allocated when None, else checked. A short, strided,
    mistyped or other-device tensor would be written out of bounds by the
    kernels, so it is refused here."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    n = 1
    for d in shape:
        n *= d
    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != torch.device(device)
            or t.dtype != dtype or t.numel() != n or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor of {n} elements on {device}")
    return t


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


# ---------------------------------------------------------------- public API
def swiglu_bwd_w_fused_workspace_size(M: int, K: int, N: int) -> int:
    return lib.swiglu_bwd_w_fused_workspace_size(M, K, N)


def swiglu_bwd_x_fused(dy, g, fc, w_g, w_fc, dx=None, dg=None, dfc=None, return_dg=False, stream=None):
    """Fused x stage: dx from dy, g, fc and the weights (dg, dfc formed on chip;
    written out too when return_dg or when passed in). Returns (dx, dg, dfc)."""
    dy, g, fc, w_g, w_fc = (_dev_bf16(t, n) for t, n in (
        (dy, "dy"), (g, "g"), (fc, "fc"), (w_g, "w_g"), (w_fc, "w_fc")))
    M, N = dy.shape
    K = w_g.shape[0]
    if g.shape != dy.shape or fc.shape != dy.shape or w_g.shape != (K, N) or w_fc.shape != (K, N):
        raise ValueError("shape mismatch: dy, g, fc [M, N]; w_g, w_fc [K, N]")
    mk = lambda t, shape: _out(t, shape, torch.bfloat16, dy.device)  # noqa: E731
    dx = mk(dx, (M, K))
    if return_dg or dg is not None or dfc is not None:
        dg, dfc = mk(dg, (M, N)), mk(dfc, (M, N))
    dev = _device_of(dy, g, fc, w_g, w_fc, dx, dg, dfc)
    _check(_call(dev, lib.swiglu_bwd_x_fused, dy.data_ptr(), g.data_ptr(), fc.data_ptr(), w_g.data_ptr(),
                 w_fc.data_ptr(), dx.data_ptr(), _ptr(dg), _ptr(dfc), M, K, N, _stream(stream, dev)),
           "swiglu_bwd_x_fused")
    return dx, dg, dfc


def swiglu_bwd_w_fused(x, dy, g, fc, dw_g=None, dw_fc=None, db_g=None, db_fc=None, workspace=None, stream=None):
    """Fused w stage: dw_g, dw_fc and db_g, db_fc from x and dy, g, fc (dg, dfc
    formed on chip). Returns (dw_g, dw_fc, db_g, db_fc)."""
    x, dy, g, fc = (_dev_bf16(t, n) for t, n in ((x, "x"), (dy, "dy"), (g, "g"), (fc, "fc")))
    M, K = x.shape
    N = dy.shape[1]
    if dy.shape != (M, N) or g.shape != (M, N) or fc.shape != (M, N):
        raise ValueError("dy, g, fc must be [M, N] with M = x.shape[0]")
    mk = lambda t, shape: _out(t, shape, torch.bfloat16, x.device)  # noqa: E731
    dw_g, dw_fc = mk(dw_g, (K, N)), mk(dw_fc, (K, N))
    db_g, db_fc = mk(db_g, (1, N)), mk(db_fc, (1, N))
    dev = _device_of(x, dy, g, fc, dw_g, dw_fc, db_g, db_fc, workspace)
    ws = _workspace(_call(dev, lib.swiglu_bwd_w_fused_workspace_size, M, K, N), x.device, workspace)
    _check(_call(dev, lib.swiglu_bwd_w_fused, x.data_ptr(), dy.data_ptr(), g.data_ptr(), fc.data_ptr(),
                 dw_g.data_ptr(), dw_fc.data_ptr(), db_g.data_ptr(), db_fc.data_ptr(), M, K, N, _ptr(ws),
                 _nbytes(ws), _stream(stream, dev)), "swiglu_bwd_w_fused")
    return dw_g, dw_fc, db_g, db_fc


SWG_INJECT_X_GEMM = 1
SWG_INJECT_FUSED_X = 2
SWG_INJECT_FUSED_W = 3
SWG_INJECT_FWD = 4


def swg_inject_stall(kernel: int, entry: int, wait_limit_cycles: int) -> None:
    """Arm a one-shot stall in the next launch of `kernel` (tests of the timeout path;
    see include/swiglu_bwd.h)."""
    _check(lib.swg_inject_stall(kernel, entry, wait_limit_cycles), "swg_inject_stall")


def swg_check(stream=None) -> None:
    """Synchronise the stream and raise if a kernel reported a barrier timeout."""
    _check(lib.swg_check(_stream(stream)), "swg_check")


def swiglu_bwd_b_workspace_size(M: int, N: int) -> int:
    return lib.swiglu_bwd_b_workspace_size(M, N)


def swiglu_bwd_w_workspace_size(M: int, K: int, N: int) -> int:
    return lib.swiglu_bwd_w_workspace_size(M, K, N)


def swiglu_bwd_kernel_count(M: int, K: int, N: int, flags: int = SWG_UNFUSED) -> int:
    """How many kernels one swiglu_bwd call with these sizes and flags launches on the current device."""
    return lib.swiglu_bwd_kernel_count(M, K, N, flags)


def swiglu_bwd_workspace_size(M: int, K: int, N: int, flags: int = SWG_UNFUSED) -> int:
    return lib.swiglu_bwd_workspace_size(M, K, N, flags)


def swiglu_bwd_b(dy, g, fc, dg=None, dfc=None, db_g=None, db_fc=None, workspace=None, stream=None):
    """b stage: returns (dg, dfc, db_g, db_fc); db_* have shape [1, N]."""
    dy, g, fc = (_dev_bf16(t, n) for t, n in ((dy, "dy"), (g, "g"), (fc, "fc")))
    M, N = dy.shape
    if g.shape != dy.shape or fc.shape != dy.shape:
        raise ValueError("dy, g, fc must have the same [M, N] shape")
    mk = lambda t, shape: _out(t, shape, torch.bfloat16, dy.device)  # noqa: E731
    dg, dfc = mk(dg, (M, N)), mk(dfc, (M, N))
    db_g, db_fc = mk(db_g, (1, N)), mk(db_fc, (1, N))
    dev = _device_of(dy, g, fc, dg, dfc, db_g, db_fc, workspace)
    ws = _workspace(_call(dev, lib.swiglu_bwd_b_workspace_size, M, N), dy.device, workspace)
    _check(_call(dev, lib.swiglu_bwd_b, dy.data_ptr(), g.data_ptr(), fc.data_ptr(), dg.data_ptr(), dfc.data_ptr(),
                 db_g.data_ptr(), db_fc.data_ptr(), M, N, _ptr(ws), _nbytes(ws), _stream(stream, dev)),
           "swiglu_bwd_b")
    return dg, dfc, db_g, db_fc


def swiglu_bwd_w(x, dg, dfc, dw_g=None, dw_fc=None, workspace=None, stream=None):
    """w stage: returns (dw_g, dw_fc), each [K, N]."""
    x, dg, dfc = (_dev_bf16(t, n) for t, n in ((x, "x"), (dg, "dg"), (dfc, "dfc")))
    M, K = x.shape
    N = dg.shape[1]
    if dg.shape != (M, N) or dfc.shape != (M, N):
        raise ValueError("dg, dfc must be [M, N] with M = x.shape[0]")
    dw_g = _out(dw_g, (K, N), torch.bfloat16, x.device, "dw_g")
    dw_fc = _out(dw_fc, (K, N), torch.bfloat16, x.device, "dw_fc")
    dev = _device_of(x, dg, dfc, dw_g, dw_fc, workspace)
    ws = _workspace(_call(dev, lib.swiglu_bwd_w_workspace_size, M, K, N), x.device, workspace)
    _check(_call(dev, lib.swiglu_bwd_w, x.data_ptr(), dg.data_ptr(), dfc.data_ptr(), dw_g.data_ptr(),
                 dw_fc.data_ptr(), M, K, N, _ptr(ws), _nbytes(ws), _stream(stream, dev)), "swiglu_bwd_w")
    return dw_g, dw_fc


def swiglu_bwd_x(dg, dfc, w_g, w_fc, dx=None, stream=None):
    """x stage: returns dx [M, K]."""
    dg, dfc, w_g, w_fc = (_dev_bf16(t, n) for t, n in ((dg, "dg"), (dfc, "dfc"), (w_g, "w_g"), (w_fc, "w_fc")))
    M, N = dg.shape
    K = w_g.shape[0]
    if dfc.shape != (M, N) or w_g.shape != (K, N) or w_fc.shape != (K, N):
        raise ValueError("shape mismatch: dg, dfc [M, N]; w_g, w_fc [K, N]")
    dx = _out(dx, (M, K), torch.bfloat16, dg.device, "dx")
    dev = _device_of(dg, dfc, w_g, w_fc, dx)
    _check(_call(dev, lib.swiglu_bwd_x, dg.data_ptr(), dfc.data_ptr(), w_g.data_ptr(), w_fc.data_ptr(),
                 dx.data_ptr(), M, K, N, _stream(stream, dev)), "swiglu_bwd_x")
    return dx


def swiglu_fwd(x, w_g, w_fc, b_g=None, b_fc=None, out: dict | None = None, stream=None) -> dict:
    """Forward: returns dict g = x W_g + b_g, fc = x W_fc + b_fc, y = SiLU(g) * fc
    (all [M, N] bf16); b_g, b_fc ([N] or [1, N]) may be None. `out` may supply
    any of g, fc, y."""
    x, w_g, w_fc = (_dev_bf16(t, n) for t, n in ((x, "x"), (w_g, "w_g"), (w_fc, "w_fc")))
    M, K = x.shape
    N = w_g.shape[1]
    if w_g.shape != (K, N) or w_fc.shape != (K, N):
        raise ValueError("shape mismatch: x [M, K]; w_g, w_fc [K, N]")
    biases = []
    for b, n in ((b_g, "b_g"), (b_fc, "b_fc")):
        if b is not None:
            b = _dev_bf16(b, n)
            if b.numel() != N:
                raise ValueError(f"{n} must have N = {N} elements")
        biases.append(b)
    out = dict(out or {})
    for k in ("g", "fc", "y"):
        out[k] = _out(out.get(k), (M, N), torch.bfloat16, x.device, k)
    dev = _device_of(x, w_g, w_fc, biases[0], biases[1], out["g"], out["fc"], out["y"])
    _check(_call(dev, lib.swiglu_fwd, x.data_ptr(), w_g.data_ptr(), w_fc.data_ptr(), _ptr(biases[0]),
                 _ptr(biases[1]), out["g"].data_ptr(), out["fc"].data_ptr(), out["y"].data_ptr(), M, K, N,
                 _stream(stream, dev)), "swiglu_fwd")
    return out


def swiglu_bwd(x, w_g, w_fc, dy, g, fc, fused: bool | None = None, return_dg: bool = True,
               out: dict | None = None, workspace=None, stream=None, accumulate: bool = False) -> dict:
    """The whole backward. Returns a dict with dx, dw_g, dw_fc, db_g, db_fc
    (and dg, dfc when return_dg). `out` may supply any of those tensors.
    fused: True (SWG_FUSED), False (SWG_UNFUSED) or None (SWG_AUTO: the library
    picks the chain measured faster for the shape).
    accumulate=True adds this call's db and dw into out's db_g, db_fc, dw_g,
    dw_fc (which must then be given) instead of overwriting them."""
    x, w_g, w_fc, dy, g, fc = (_dev_bf16(t, n) for t, n in (
        (x, "x"), (w_g, "w_g"), (w_fc, "w_fc"), (dy, "dy"), (g, "g"), (fc, "fc")))
    M, K = x.shape
    N = w_g.shape[1]
    for t, n, shp in ((w_fc, "w_fc", (K, N)), (dy, "dy", (M, N)), (g, "g", (M, N)), (fc, "fc", (M, N)),
                      (w_g, "w_g", (K, N))):
        if tuple(t.shape) != shp:
            raise ValueError(f"{n} must have shape {shp}, got {tuple(t.shape)}")
    out = dict(out or {})
    if accumulate and any(out.get(k) is None for k in ("dw_g", "dw_fc", "db_g", "db_fc")):
        raise ValueError("accumulate=True needs dw_g, dw_fc, db_g and db_fc in `out`")
    shapes = dict(dx=(M, K), dw_g=(K, N), dw_fc=(K, N), db_g=(1, N), db_fc=(1, N))
    if return_dg or out.get("dg") is not None or out.get("dfc") is not None:
        shapes.update(dg=(M, N), dfc=(M, N))
    for k, shp in shapes.items():
        out[k] = _out(out.get(k), shp, torch.bfloat16, x.device, k)
    flags = (SWG_AUTO if fused is None else SWG_FUSED if fused else SWG_UNFUSED) | (SWG_ACCUMULATE if accumulate else 0)
    ws_flags = flags | (SWG_WS_DG_GIVEN if return_dg else 0)
    dev = _device_of(x, w_g, w_fc, dy, g, fc, workspace, *out.values())
    ws = _workspace(_call(dev, lib.swiglu_bwd_workspace_size, M, K, N, ws_flags), x.device, workspace)
    _check(_call(dev, lib.swiglu_bwd, x.data_ptr(), w_g.data_ptr(), w_fc.data_ptr(), dy.data_ptr(), g.data_ptr(),
                 fc.data_ptr(), _ptr(out.get("dg")), _ptr(out.get("dfc")), out["dx"].data_ptr(),
                 out["dw_g"].data_ptr(), out["dw_fc"].data_ptr(), out["db_g"].data_ptr(),
                 out["db_fc"].data_ptr(), M, K, N, flags, _ptr(ws), _nbytes(ws), _stream(stream, dev)),
           "swiglu_bwd")
    return out


def swish_grad(grad, x, scale=None, grad_x=None, stream=None):
    """SwishGrad: grad_x = grad * sigma(beta x) * (1 + beta x (1 - sigma(beta x))); beta = scale or 1.0."""
    if not (isinstance(grad, torch.Tensor) and isinstance(x, torch.Tensor) and grad.is_cuda and x.is_cuda):
        raise TypeError("grad and x must be CUDA tensors")
    if grad.dtype != x.dtype or grad.shape != x.shape:
        raise ValueError("grad and x must have the same dtype and shape")
    if grad.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {grad.dtype}")
    grad, x = grad.contiguous(), x.contiguous()
    grad_x = _out(grad_x, tuple(grad.shape), grad.dtype, grad.device, "grad_x")
    sc = None if scale is None else ctypes.byref(ctypes.c_float(scale))
    dev = _device_of(grad, x, grad_x)
    _check(_call(dev, lib.swish_grad, grad.data_ptr(), x.data_ptr(), sc, grad_x.data_ptr(), grad.numel(),
                 _DTYPE[grad.dtype], _stream(stream, dev)), "swish_grad")
    return grad_x


SWG_ACT = {"silu": 0, "gelu": 1, "hardswish": 2}


def act_grad(grad, x, act: str, grad_x=None, stream=None):
    """Activation gradient grad * f'(x) for act in "silu", "gelu", "hardswish"
    (fp32/fp16/bf16, any shape, treated as 1-D)."""
    if act not in SWG_ACT:
        raise ValueError(f"act must be one of {sorted(SWG_ACT)}")
    if not (isinstance(grad, torch.Tensor) and isinstance(x, torch.Tensor) and grad.is_cuda and x.is_cuda):
        raise TypeError("grad and x must be CUDA tensors")
    if grad.dtype != x.dtype or grad.shape != x.shape:
        raise ValueError("grad and x must have the same dtype and shape")
    if grad.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {grad.dtype}")
    grad, x = grad.contiguous(), x.contiguous()
    grad_x = _out(grad_x, tuple(grad.shape), grad.dtype, grad.device, "grad_x")
    dev = _device_of(grad, x, grad_x)
    _check(_call(dev, lib.act_grad, grad.data_ptr(), x.data_ptr(), SWG_ACT[act], grad_x.data_ptr(), grad.numel(),
                 _DTYPE[grad.dtype], _stream(stream, dev)), "act_grad")
    return grad_x


def swiglu_bwd_host_workspace_size(M: int, K: int, N: int) -> int:
    return int(lib.swiglu_bwd_host_workspace_size(M, K, N))


def swiglu_bwd_host(x, w_g, w_fc, dy, g, fc, out: dict | None = None, workspace=None, stream=None) -> dict:
    """Whole fused backward with every tensor in host memory (bf16 CPU tensors; pinned ones let the
    copies overlap the compute). Returns host tensors dx, dw_g, dw_fc, db_g, db_fc (pinned when
    allocated here); they are complete once `stream` (default: the current CUDA stream) has run."""
    ins = dict(x=x, w_g=w_g, w_fc=w_fc, dy=dy, g=g, fc=fc)
    for k, t in ins.items():
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{k} must be a bf16 CPU tensor")
    ins = {k: t.contiguous() for k, t in ins.items()}
    M, K = ins["x"].shape
    N = ins["w_g"].shape[1]
    if out is None:
        out = {}
    for k, t in ins.items():
        want = {"x": M * K, "w_g": K * N, "w_fc": K * N, "dy": M * N, "g": M * N, "fc": M * N}[k]
        if t.numel() != want:
            raise ValueError(f"{k} must have {want} elements for M={M}, K={K}, N={N}")
    shapes = dict(dx=(M, K), dw_g=(K, N), dw_fc=(K, N), db_g=(1, N), db_fc=(1, N))
    for k, t in out.items():
        shp = shapes[k]
        # the library copies into these buffers: a short or strided one would be overrun
        if (not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16
                or t.numel() != shp[0] * shp[1] or not t.is_contiguous()):
            raise ValueError(f"out[{k!r}] must be a contiguous bf16 CPU tensor of {shp[0] * shp[1]} elements")
    for k, shp in shapes.items():
        if k not in out:
            out[k] = torch.empty(shp, dtype=torch.bfloat16, pin_memory=True)
    # the device is the workspace's when one is given, else the current one
    dev = workspace.device if workspace is not None else torch.device("cuda", torch.cuda.current_device())
    if not dev.type == "cuda":
        raise ValueError("workspace must be a CUDA tensor")
    ws = _workspace(_call(dev, swiglu_bwd_host_workspace_size, M, K, N), dev, workspace)
    _check(_call(dev, lib.swiglu_bwd_host, *(ins[k].data_ptr() for k in ("x", "w_g", "w_fc", "dy", "g", "fc")),
                 *(out[k].data_ptr() for k in ("dx", "dw_g", "dw_fc", "db_g", "db_fc")),
                 M, K, N, _ptr(ws), _nbytes(ws), _stream(stream, dev)), "swiglu_bwd_host")
    return out


def group_norm_bwd_workspace_size(N: int, C: int, HxW: int, G: int) -> int:
    return int(lib.group_norm_bwd_workspace_size(N, C, HxW, G))


def group_norm_bwd(dy, x, num_groups: int, gamma=None, eps: float = 1e-5, params: bool = True,
                   dx=None, dgamma=None, dbeta=None, workspace=None, stream=None):
    """GroupNorm backward for x, dy of shape [N, C, *spatial] (fp32/fp16/bf16):
    returns (dx, dgamma, dbeta); dgamma and dbeta are None when params is False.
    gamma [C] (same dtype) may be None (= ones). Statistics are recomputed from x."""
    if not (isinstance(dy, torch.Tensor) and isinstance(x, torch.Tensor) and dy.is_cuda and x.is_cuda):
        raise TypeError("dy and x must be CUDA tensors")
    if dy.dtype != x.dtype or dy.shape != x.shape:
        raise ValueError("dy and x must have the same dtype and shape")
    if x.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {x.dtype}")
    if x.dim() < 2:
        raise ValueError("x must be [N, C, *spatial]")
    N, C = x.shape[0], x.shape[1]
    HxW = 1
    for d in x.shape[2:]:
        HxW *= d
    if gamma is not None:
        if not (isinstance(gamma, torch.Tensor) and gamma.is_cuda) or gamma.dtype != x.dtype or gamma.numel() != C:
            raise ValueError("gamma must be a CUDA tensor of C elements with x's dtype")
        gamma = gamma.contiguous()
    dy, x = dy.contiguous(), x.contiguous()
    dx = _out(dx, tuple(x.shape), x.dtype, x.device, "dx")
    if params:
        dgamma = _out(dgamma, (C,), x.dtype, x.device, "dgamma")
        dbeta = _out(dbeta, (C,), x.dtype, x.device, "dbeta")
        ws = _workspace(group_norm_bwd_workspace_size(N, C, HxW, num_groups), x.device, workspace)
    else:
        dgamma = dbeta = ws = None
    dev = _device_of(dy, x, gamma, dx, dgamma, dbeta, ws)
    _check(_call(dev, lib.group_norm_bwd, dy.data_ptr(), x.data_ptr(), _ptr(gamma), dx.data_ptr(), _ptr(dgamma),
                 _ptr(dbeta), N, C, HxW, num_groups, float(eps), _DTYPE[x.dtype], _ptr(ws), _nbytes(ws),
                 _stream(stream, dev)), "group_norm_bwd")
    return dx, dgamma, dbeta


def swiglu_bwd_b_noalloc(dy, g, fc, dg=None, dfc=None, db_g=None, db_fc=None, stream=None):
    """b stage without a workspace: the column partials use a fixed array
    inside the library, so the call itself allocates nothing on the device
    (outputs not passed in are still created here with torch.empty). Calls
    must not overlap on the GPU; see include/swiglu_bwd.h."""
    dy, g, fc = (_dev_bf16(t, n) for t, n in ((dy, "dy"), (g, "g"), (fc, "fc")))
    M, N = dy.shape
    if g.shape != dy.shape or fc.shape != dy.shape:
        raise ValueError("dy, g, fc must have the same [M, N] shape")
    mk = lambda t, shape: _out(t, shape, torch.bfloat16, dy.device)  # noqa: E731
    dg, dfc = mk(dg, (M, N)), mk(dfc, (M, N))
    db_g, db_fc = mk(db_g, (1, N)), mk(db_fc, (1, N))
    dev = _device_of(dy, g, fc, dg, dfc, db_g, db_fc)
    _check(_call(dev, lib.swiglu_bwd_b_noalloc, dy.data_ptr(), g.data_ptr(), fc.data_ptr(), dg.data_ptr(),
                 dfc.data_ptr(), db_g.data_ptr(), db_fc.data_ptr(), M, N, _stream(stream, dev)),
           "swiglu_bwd_b_noalloc")
    return dg, dfc, db_g, db_fc
