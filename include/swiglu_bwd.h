/*
 * swiglu_bwd.h -- C ABI of the GB300 (sm_103a) SwiGLU-FFN backward, SwishGrad,
 * the sibling activation gradients and the GroupNorm backward.
 *
 * Operations (sources are web pages; each function cites the section it follows):
 *   [P1] "PyPTO-Gym in practice: the fused SwiGLU backward operator"
 *        (hnwysp.cn/news/34787)
 *   [P2] "SwishGrad in CANN ops-nn: principle, implementation and the
 *        aclnnSwishBackward guide" (bhfrc.com/news/37500)
 *   [P3] "Beyond automatic differentiation: efficient custom backward
 *        operators in Ascend C" (cann.csdn.net): activation gradients and the
 *        GroupNorm backward
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, row-major, contiguous, on the current CUDA device.
 *   SwiGLU tensors are bf16 (2 bytes, stored as uint16 bit patterns).
 *   Shapes follow [P1] "Kernel signatures": x [M,K]; w_g, w_fc [K,N];
 *   dy, g, fc, dg, dfc [M,N]; db_g, db_fc [1,N]; dw_g, dw_fc [K,N]; dx [M,K].
 * - Ownership: the caller owns every buffer, including the workspace, whose
 *   size comes from the matching *_workspace_size query (the two-phase model of
 *   [P2] section 3.2). The library keeps no per-call state and allocates no
 *   device memory; a 4-byte device status word (see swg_check) is its only
 *   module-level device state.
 * - Streams: every call is asynchronous on `stream` (NULL = legacy default
 *   stream), like aclnnSwishBackward ([P2] section 3.4). Argument errors are
 *   returned synchronously with nothing launched. A failed launch returns
 *   SWG_ERR_CUDA.
 * - Dynamic M ([P1] "Dynamic axis M"): any M >= 0 without recompilation; a
 *   tail of M that does not fill a tile is handled inside the kernels.
 *   K and N must be positive multiples of 8 (16-byte rows for TMA); other
 *   values return SWG_ERR_UNSUPPORTED. Base pointers of SwiGLU tensors and of
 *   the workspace must be 16-byte aligned (SWG_ERR_UNSUPPORTED otherwise).
 * - Empty calls: M == 0 (or n == 0) launches no element-wise work ([P2]
 *   section 3.5, empty-tensor short circuit); outputs that are sums over the
 *   M rows (db_*, dw_*) are still written, as zeros. Pointers of empty
 *   tensors (those with an M dimension when M == 0, all of swish_grad's
 *   when n == 0) may be NULL.
 * - Outputs are OVERWRITTEN. [P1] asks callers to zero db/dw and accumulates
 *   into them; overwriting gives the same values without the zeroing.
 * - Outputs must not overlap inputs or each other (SWG_ERR_PARAM_INVALID when
 *   an overlap is detected from the pointer ranges). Exception: swish_grad's
 *   grad_x may alias grad or x exactly.
 * - Arithmetic: bf16 inputs are widened to fp32; element-wise math, sums and
 *   tensor-core accumulation are fp32; each output is rounded once to bf16,
 *   round-to-nearest-even ([P1] "Dtype conversion flow": bf16 storage, fp32
 *   compute; [P2] section 2.4, CAST_RINT).
 */
#ifndef SWIGLU_BWD_H
#define SWIGLU_BWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* swg_stream_t;

typedef enum {
  SWG_OK = 0,
  SWG_ERR_NULLPTR = 1,       /* a required pointer is NULL ([P2] 3.3: ACLNN_ERR_PARAM_NULLPTR) */
  SWG_ERR_PARAM_INVALID = 2, /* bad dtype / negative size / overlapping buffers
                                ([P2] 3.3: ACLNN_ERR_PARAM_INVALID) */
  SWG_ERR_UNSUPPORTED = 3,   /* K or N not a positive multiple of 8, misaligned
                                pointer, or the current device is not sm_103 */
  SWG_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than the size query */
  SWG_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
  SWG_ERR_TIMEOUT = 6        /* a kernel gave up waiting on one of its pipeline barriers */
} swg_status;

typedef enum { SWG_F32 = 0, SWG_F16 = 1, SWG_BF16 = 2 } swg_dtype;

/* activations whose gradient act_grad computes */
typedef enum { SWG_ACT_SILU = 0, SWG_ACT_GELU = 1, SWG_ACT_HARDSWISH = 2 } swg_act;

/* flags for swiglu_bwd */
#define SWG_UNFUSED 0u /* b stage, then the w and x GEMMs on the stored dg, dfc */
#define SWG_FUSED 1u   /* the GEMMs recompute dg, dfc from dy, g, fc in their
                          operand producer; dg, dfc never round-trip HBM */
/* Accumulate mode ([P1] "Kernel signatures": the pages' b and w kernels add
 * their db and dw into outputs the caller has zeroed, so that several
 * micro-batches can be summed). With SWG_ACCUMULATE, db_g, db_fc, dw_g and
 * dw_fc are read and replaced by bf16(old + this call's sum): the fp32 (db:
 * fp64) sum and the old value are added before the single rounding. dx, dg and
 * dfc are still overwritten. With M == 0 the four outputs are left unchanged.
 * Without the flag every output is overwritten (the same result as the pages'
 * zero-then-accumulate on zeroed outputs). */
#define SWG_ACCUMULATE 2u
/* The library chooses the chain (replaces SWG_FUSED / SWG_UNFUSED): fused when
 * K <= 512 and M >= 32768, unfused otherwise -- the faster one in measurements
 * on GB300 (fused: 0.80 vs 1.07 ms at M=220000 K=512 N=1024 and faster from
 * M = 65537 on at K=512; unfused: faster at M <= 4097, and 5.48 vs 6.85 ms at
 * the LLM FFN shape M=16384 K=4096 N=14336, where the fused kernels would form
 * dg, dfc eight times each). The workspace query resolves it the same way. */
#define SWG_AUTO 4u

/* Human-readable name of a status code (static storage, never NULL). */
const char* swg_status_string(swg_status s);

/* Synchronises `stream`, then reports and clears the device status word that
 * kernels set when a bounded pipeline wait runs out (SWG_ERR_TIMEOUT), or
 * returns SWG_ERR_CUDA if the stream reports an error. SWG_OK otherwise. */
swg_status swg_check(swg_stream_t stream);

/* ---- fault injection for tests of the timeout path ------------------------------
 * No counterpart on the pages. Every pipeline wait in the tcgen05 kernels is a
 * bounded spin (about 2 s); this arms a one-shot fault for the NEXT launch of
 * one kernel by this process, so that a test can see a wait run out without
 * faulting or hanging the GPU: that launch's operand producer stops issuing
 * copies before ring entry `entry` (nothing is left in flight), and each of its
 * waits gives up after `wait_limit_cycles` SM clock cycles. The consumer's wait
 * on the missing entry then runs out; the kernel sets the status word, stops,
 * waits (bounded) for the work it did issue, frees its tensor memory and
 * returns. That launch's outputs are incomplete; swg_check() then reports
 * SWG_ERR_TIMEOUT and clears the word, and later calls run normally.
 *   kernel: SWG_INJECT_X_GEMM (the x stage's GEMM, swiglu_bwd_x and the
 *           unfused swiglu_bwd), SWG_INJECT_FUSED_X (the fused x kernel,
 *           swiglu_bwd_x_fused and the fused swiglu_bwd) or SWG_INJECT_FUSED_W
 *           (the fused w kernel on CTA pairs, swiglu_bwd_w_fused and the fused
 *           swiglu_bwd: both CTAs' producers stop at the entry) or SWG_INJECT_FWD
 *           (the forward on CTA pairs, swiglu_fwd: both producers stop).
 * SWG_INJECT_NONE disarms an armed, unused injection (entry and limit are then
 * ignored); a later call replaces it. Returns SWG_ERR_PARAM_INVALID for another
 * kernel, entry < 0 or a limit below 1024 cycles. For tests only. */
typedef enum {
  SWG_INJECT_NONE = 0,
  SWG_INJECT_X_GEMM = 1,
  SWG_INJECT_FUSED_X = 2,
  SWG_INJECT_FUSED_W = 3,
  SWG_INJECT_FWD = 4
} swg_inject_kernel;
swg_status swg_inject_stall(swg_inject_kernel kernel, int64_t entry, int64_t wait_limit_cycles);

/* ---- b stage -----------------------------------------------------------------
 * [P1] "Algorithm overview and formulas" items 1-2; "Kernel signatures",
 * fused_swiglu_bwd_b_kernel(dy, g, fc, dg, dfc, db_g, db_fc):
 *   s = sigma(g);  dg = dy * fc * s * (1 + g * (1 - s));  dfc = dy * g * s;
 *   db_g[n] = sum_m dg[m,n];  db_fc[n] = sum_m dfc[m,n].
 * The column sums are taken over the fp32 dg, dfc (before bf16 rounding), as
 * fp32 per-block partials reduced in a fixed order (deterministic).
 * Inputs: dy, g, fc [M,N]. Outputs: dg, dfc [M,N]; db_g, db_fc [1,N].
 * Workspace: swiglu_bwd_b_workspace_size(M, N) bytes, 16-byte aligned. */
size_t swiglu_bwd_b_workspace_size(int64_t M, int64_t N);
swg_status swiglu_bwd_b(const void* dy, const void* g, const void* fc,
                        void* dg, void* dfc, void* db_g, void* db_fc,
                        int64_t M, int64_t N, void* workspace, size_t workspace_bytes,
                        swg_stream_t stream);

/* ---- b stage without a workspace ----------------------------------------------
 * No counterpart on the pages: an addition for callers that cannot allocate
 * device memory and cannot hold a workspace between calls (for example a host
 * framework whose memory pool owns all of device memory, or a loop that cannot
 * afford cudaMalloc's implicit synchronisation). Same inputs, outputs and
 * results as swiglu_bwd_b; the fp32 column partials live in a 4 MiB array
 * compiled into the library (SWG_NOALLOC_SCRATCH_BYTES), held by every GPU that
 * loads the library until the process exits. Nothing is allocated.
 * - Limit: the partials must fit the array, which holds for every M when
 *   N <= 524288; larger shapes return SWG_ERR_WORKSPACE with nothing launched.
 * - Each call looks up the array's device address on the current device
 *   (so calls stay valid across a cudaDeviceReset); the first call on a
 *   device also loads the library's device code there, so make that first
 *   call before any stream capture.
 * - Every call shares the array and it keeps the last call's contents (no
 *   call needs it zeroed). Calls that overlap on the GPU, e.g. on two streams
 *   at once, race on it and give wrong db; serialise them. */
#define SWG_NOALLOC_SCRATCH_BYTES (4u << 20)
swg_status swiglu_bwd_b_noalloc(const void* dy, const void* g, const void* fc,
                                void* dg, void* dfc, void* db_g, void* db_fc,
                                int64_t M, int64_t N, swg_stream_t stream);

/* ---- w stage -----------------------------------------------------------------
 * [P1] item 3; fused_swiglu_bwd_w_kernel(x, dg, dfc, dw_g, dw_fc):
 *   dw_g = x^T dg;  dw_fc = x^T dfc      (x [M,K]; dg, dfc [M,N]; dw_* [K,N])
 * One tcgen05 GEMM launch covers both outputs; the reduction runs over M and
 * may be split over M into fp32 partials (workspace) that a second kernel sums
 * in a fixed order before the single bf16 rounding.
 * Workspace: swiglu_bwd_w_workspace_size(M, K, N) bytes (may be 0). */
size_t swiglu_bwd_w_workspace_size(int64_t M, int64_t K, int64_t N);
swg_status swiglu_bwd_w(const void* x, const void* dg, const void* dfc,
                        void* dw_g, void* dw_fc, int64_t M, int64_t K, int64_t N,
                        void* workspace, size_t workspace_bytes, swg_stream_t stream);

/* ---- x stage -----------------------------------------------------------------
 * [P1] item 4; fused_swiglu_bwd_x_kernel(dg, dfc, w_g, w_fc, dx):
 *   dx = dg W_g^T + dfc W_fc^T           (dx [M,K])
 * computed as one GEMM [dg | dfc] [W_g | W_fc]^T with reduction length 2N;
 * no workspace. */
swg_status swiglu_bwd_x(const void* dg, const void* dfc, const void* w_g, const void* w_fc,
                        void* dx, int64_t M, int64_t K, int64_t N, swg_stream_t stream);

/* ---- fused stages -------------------------------------------------------------
 * The b-stage math of [P1] item 1 runs inside the GEMMs' operand producer:
 * dg, dfc are computed from dy, g, fc tile by tile in shared memory, rounded to
 * bf16 exactly as the b stage stores them, and fed to the tensor cores; they
 * are never written to or read back from HBM (the recompute-instead-of-store
 * principle).
 *
 * swiglu_bwd_x_fused: dx = dg W_g^T + dfc W_fc^T ([P1] item 4) from dy, g, fc
 *   [M,N] and w_g, w_fc [K,N]. dg, dfc [M,N] are optional outputs (NULL to
 *   skip; both or neither). No workspace.
 * swiglu_bwd_w_fused: dw_g = x^T dg, dw_fc = x^T dfc ([P1] item 3) and the
 *   column sums db_g, db_fc ([P1] item 2) from x [M,K] and dy, g, fc.
 *   Workspace: split-M fp32 partials of dw and db,
 *   swiglu_bwd_w_fused_workspace_size(M, K, N) bytes.
 * Same shape, alignment, overlap and error rules as the unfused stages. */
swg_status swiglu_bwd_x_fused(const void* dy, const void* g, const void* fc,
                              const void* w_g, const void* w_fc, void* dx, void* dg, void* dfc,
                              int64_t M, int64_t K, int64_t N, swg_stream_t stream);
size_t swiglu_bwd_w_fused_workspace_size(int64_t M, int64_t K, int64_t N);
swg_status swiglu_bwd_w_fused(const void* x, const void* dy, const void* g, const void* fc,
                              void* dw_g, void* dw_fc, void* db_g, void* db_fc,
                              int64_t M, int64_t K, int64_t N,
                              void* workspace, size_t workspace_bytes, swg_stream_t stream);

/* ---- forward ----------------------------------------------------------------
 * [P1] "Operator background" (the forward whose outputs the backward takes):
 *   g  = x W_g + b_g,   fc = x W_fc + b_fc      (g, fc [M,N])
 *   y  = SiLU(g) * fc = g * sigma(g) * fc        (y [M,N])
 * x [M,K], w_g/w_fc [K,N], b_g/b_fc [N] (NULL: no bias), all bf16 row-major.
 * One tcgen05 GEMM launch (fp32 accumulation) computes both products; g, fc
 * are formed in fp32 with the bias and y from those fp32 values; each output
 * is rounded once to bf16 (round to nearest even). K must be positive
 * (K == 0: SWG_ERR_UNSUPPORTED); M == 0 or N == 0: nothing is launched.
 * Outputs must not overlap the inputs or each other (SWG_ERR_PARAM_INVALID);
 * no workspace. */
swg_status swiglu_fwd(const void* x, const void* w_g, const void* w_fc,
                      const void* b_g, const void* b_fc, void* g, void* fc, void* y,
                      int64_t M, int64_t K, int64_t N, swg_stream_t stream);

/* ---- whole backward ----------------------------------------------------------
 * [P1] "Kernel overview and call chain": b, then w and x on b's dg, dfc.
 * flags: SWG_UNFUSED, SWG_FUSED or SWG_AUTO, optionally | SWG_ACCUMULATE.
 * dg, dfc are optional outputs: pass NULL to skip them. With SWG_UNFUSED and
 * NULL dg/dfc, the workspace holds them (4*M*N bytes more). With SWG_FUSED the
 * call runs the work of swiglu_bwd_w_fused and swiglu_bwd_x_fused: the w and x
 * GEMMs compute dg, dfc tile by tile in shared memory from dy, g, fc; their
 * operands are the bf16 roundings of the fp32 dg, dfc, exactly as in the
 * unfused chain. When the w stage leaves SMs free and the x stage needs more
 * than one wave of tiles, the x stage's last tiles run beside the w stage on a
 * library-owned side stream (forked from and joined back into `stream` within
 * the call, so the call stays ordered on `stream` and can be captured in a CUDA
 * graph) and the rest after it; the w stage's split reduction then also runs on
 * the side stream, in blocks that fit beside the x stage's persistent wave.
 * Every output is bit-identical to the two stage calls.
 * Workspace: swiglu_bwd_workspace_size(M, K, N, flags) bytes; with non-NULL
 * dg/dfc the smaller figure swiglu_bwd_workspace_size(M, K, N, flags |
 * SWG_WS_DG_GIVEN) suffices. */
#define SWG_WS_DG_GIVEN 0x100u
size_t swiglu_bwd_workspace_size(int64_t M, int64_t K, int64_t N, unsigned flags);
swg_status swiglu_bwd(const void* x, const void* w_g, const void* w_fc,
                      const void* dy, const void* g, const void* fc,
                      void* dg, void* dfc, void* dx, void* dw_g, void* dw_fc,
                      void* db_g, void* db_fc, int64_t M, int64_t K, int64_t N,
                      unsigned flags, void* workspace, size_t workspace_bytes,
                      swg_stream_t stream);

/* The number of kernels one swiglu_bwd(..., M, K, N, flags, ...) call launches
 * on the current device: 0 for a call that launches none (M == 0 clears its
 * outputs with memsets; K or N == 0; invalid arguments). Launches nothing; for
 * launch accounting and profiling. */
int swiglu_bwd_kernel_count(int64_t M, int64_t K, int64_t N, unsigned flags);

/* ---- whole fused backward from host buffers ------------------------------------
 * The whole backward of swiglu_bwd(..., SWG_FUSED, ...) (dx, dw_g, dw_fc, db_g,
 * db_fc; dg and dfc are not produced) with every tensor argument in HOST
 * memory, same shapes and layouts as swiglu_bwd. Page-locked host buffers
 * (cudaHostAlloc / cudaHostRegister) let the copies overlap: M is cut into
 * chunks of 32768 rows or more and a short last one (at least 16384 rows);
 * while one chunk is computed, the next chunk's
 * rows are copied in and the previous chunk's dx is copied out, on two
 * internal streams ordered against `stream` with events. dw and db are
 * reduced once over every chunk's fp32 partials (one rounding, as in
 * swiglu_bwd). `workspace` is DEVICE memory of at least
 * swiglu_bwd_host_workspace_size(M, K, N) bytes, 16-byte aligned (it holds
 * two chunks of inputs and of dx, W, the outputs and the partials: about
 * 0.8 GB at M = 220000, K = 512, N = 1024). The call is asynchronous on
 * `stream`: the host outputs are complete once the work enqueued on `stream`
 * up to this call has finished (e.g. after cudaStreamSynchronize). Outputs
 * are overwritten (no SWG_ACCUMULATE). Errors as swiglu_bwd, plus
 * SWG_ERR_WORKSPACE for a missing or short workspace. */
size_t swiglu_bwd_host_workspace_size(int64_t M, int64_t K, int64_t N);
swg_status swiglu_bwd_host(const void* x, const void* w_g, const void* w_fc,
                           const void* dy, const void* g, const void* fc,
                           void* dx, void* dw_g, void* dw_fc, void* db_g, void* db_fc,
                           int64_t M, int64_t K, int64_t N, void* workspace,
                           size_t workspace_bytes, swg_stream_t stream);

/* ---- SwishGrad ---------------------------------------------------------------
 * [P2] section 1.2: grad_x = grad * sigma(beta x) * (1 + beta x (1 - sigma(beta x))),
 * beta = *scale, or 1.0 when scale is NULL ([P2] 3.5). grad, x, grad_x hold n
 * elements of `dtype` (fp32 / fp16 / bf16; any shape, treated as 1-D; any
 * alignment; any n >= 0). Math is fp32; fp16/bf16 results are rounded to
 * nearest even ([P2] 2.4, CAST_RINT). grad_x may alias grad or x exactly.
 * No workspace ([P2]'s workspace query returns 0 for this op as well). */
swg_status swish_grad(const void* grad, const void* x, const float* scale, void* grad_x,
                      int64_t n, swg_dtype dtype, swg_stream_t stream);

/* ---- sibling activation gradients -------------------------------------------
 * The Ascend C backward blog post names GELU and HardSwish as the next
 * activations to give a hand-written backward, and SiluGrad as SwishGrad's
 * sibling; the pages give no formula for them, so the standard definitions
 * are used: grad_x = grad * f'(x), fp32 math, fp16/bf16 rounded once (RNE).
 *   SWG_ACT_SILU:      f(x) = x sigma(x) -- identical to swish_grad with
 *                      scale 1.0, bit for bit
 *   SWG_ACT_GELU:      f(x) = x Phi(x) (exact, erf form);
 *                      f'(x) = Phi(x) + x phi(x)
 *   SWG_ACT_HARDSWISH: f(x) = x min(max(x + 3, 0), 6) / 6;
 *                      f'(x) = 0 (x <= -3), x/3 + 1/2 (-3 < x < 3), 1 (x >= 3),
 *                      the kinks as in PyTorch's autograd
 * Same arguments, layout, aliasing and error rules as swish_grad (an unknown
 * act is SWG_ERR_PARAM_INVALID). */
swg_status act_grad(const void* grad, const void* x, swg_act act, void* grad_x,
                    int64_t n, swg_dtype dtype, swg_stream_t stream);

/* ---- GroupNorm backward -----------------------------------------------------
 * [P3] GroupNorm section (revised version 3.1-3.2): for x, dy of shape
 * [N, C, HxW] (NCHW, spatial dimensions flattened, contiguous) split into G
 * groups of C/G consecutive channels per sample, m = (C/G) HxW elements per
 * group, mu and the biased variance var of each group recomputed from x,
 * rstd = 1/sqrt(var + eps), x_hat = (x - mu) rstd:
 *   dx       = rstd (gamma_c dy - sum(gamma dy)/m - x_hat sum(gamma dy x_hat)/m),
 *   dgamma_c = sum over samples and positions of dy x_hat,
 *   dbeta_c  = sum over samples and positions of dy
 * (the pages give dx; dgamma and dbeta are the standard parameter gradients).
 * gamma [C] may be NULL (gamma = 1). dgamma, dbeta [C] are optional outputs
 * (NULL: not computed); when either is given, `workspace` must hold at least
 * group_norm_bwd_workspace_size(N, C, HxW, G) bytes (16-byte aligned), else
 * SWG_ERR_WORKSPACE; without them the workspace is unused and may be NULL.
 * All tensors share `dtype` (fp32 / fp16 / bf16), aligned to their element size
 * (SWG_ERR_UNSUPPORTED otherwise); 16-byte aligned groups take the bulk-copy
 * path, others plain loads. Math is fp32, sums in a fixed order (dgamma and
 * dbeta: each sample's partials added in fp32, the samples in fp64); each
 * output is rounded once (RNE); results are bitwise reproducible.
 * Errors: G < 1, C not a multiple of G, a negative size or a negative / NaN eps
 * -> SWG_ERR_PARAM_INVALID; N G >= 2^28 or N C HxW >= 2^60 -> SWG_ERR_UNSUPPORTED; x, dy or dx NULL
 * with N C HxW > 0 -> SWG_ERR_NULLPTR; outputs overlapping inputs or each other
 * -> SWG_ERR_PARAM_INVALID. Empty (N C HxW == 0): no dx work; dgamma, dbeta
 * (sums over nothing) are written as zeros. */
size_t group_norm_bwd_workspace_size(int64_t N, int64_t C, int64_t HxW, int64_t G);
swg_status group_norm_bwd(const void* dy, const void* x, const void* gamma, void* dx,
                          void* dgamma, void* dbeta, int64_t N, int64_t C, int64_t HxW,
                          int64_t G, float eps, swg_dtype dtype, void* workspace,
                          size_t workspace_bytes, swg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_BWD_H */
