"""GB300 (sm_103a) SwiGLU-FFN backward, SwishGrad, activation gradients and
the GroupNorm backward.

The compute runs in hand-written CUDA kernels behind the C ABI of
include/swiglu_bwd.h; this package is the thin Python binding over it.
"""

from ._binding import (  # noqa: F401
    EXPORTS,
    act_grad,
    group_norm_bwd,
    group_norm_bwd_workspace_size,
    LIB_PATH,
    SWG_ACCUMULATE,
    SWG_AUTO,
    SWG_FUSED,
    SWG_UNFUSED,
    SwgError,
    status_string,
    swg_check,
    swg_inject_stall,
    SWG_INJECT_FUSED_W,
    SWG_INJECT_FWD,
    SWG_INJECT_FUSED_X,
    SWG_INJECT_X_GEMM,
    swiglu_bwd,
    swiglu_bwd_b,
    swiglu_bwd_b_noalloc,
    swiglu_bwd_b_workspace_size,
    swiglu_bwd_host,
    swiglu_bwd_host_workspace_size,
    swiglu_bwd_kernel_count,
    swiglu_bwd_w,
    swiglu_bwd_w_workspace_size,
    swiglu_bwd_workspace_size,
    swiglu_bwd_w_fused,
    swiglu_bwd_w_fused_workspace_size,
    swiglu_bwd_x,
    swiglu_bwd_x_fused,
    swiglu_fwd,
    swish_grad,
)
