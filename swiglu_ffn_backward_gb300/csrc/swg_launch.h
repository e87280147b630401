// Internal host-side launchers (C++ linkage). The C ABI in include/swiglu_bwd.h
// validates arguments and then calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace swg {

// ---- SwishGrad: dtype 0 = f32, 1 = f16, 2 = bf16
cudaError_t launch_swish_grad(const void* grad, const void* x, float beta, void* grad_x, int64_t n, int dtype,
                              cudaStream_t stream);
// activation gradients grad * f'(x): act 0 = SiLU (SwishGrad with beta 1), 1 = GELU (exact), 2 = HardSwish
cudaError_t launch_act_grad(const void* grad, const void* x, int act, void* grad_x, int64_t n, int dtype,
                            cudaStream_t stream);

// ---- b stage
struct BPlan {
  int64_t rows_per_chunk;  // rows of M per CTA row-chunk (multiple of 8)
  int64_t chunks;          // number of row chunks = fp32 partial rows in the workspace
};
BPlan b_plan(int64_t M, int64_t N);
size_t b_workspace_bytes(int64_t M, int64_t N);
// dg/dfc may be null (then only the column sums are produced)
// accumulate: db_g, db_fc += the column sums (one rounding of old + new); default: overwrite
cudaError_t launch_b_stage(const uint16_t* dy, const uint16_t* g, const uint16_t* fc, uint16_t* dg, uint16_t* dfc,
                           uint16_t* db_g, uint16_t* db_fc, int64_t M, int64_t N, void* ws, cudaStream_t stream,
                           bool accumulate = false);
// db from fp32 partials [chunks][2N] -> bf16 db_g, db_fc (fixed order)
cudaError_t launch_db_reduce(const float* partials, int64_t chunks, int64_t N, uint16_t* db_g, uint16_t* db_fc,
                             cudaStream_t stream, bool accumulate = false);
// 3-D tensor-map encoding (dims/strides innermost first; strides[i] is the byte stride of dim i+1)
bool encode_tmap_3d_bf16(CUtensorMap* tm, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                         const uint32_t box[3], int swizzle_bytes);

// ---- tcgen05 GEMMs
struct WPlan {
  int64_t splits;     // M split count for the dw reduction
  int64_t kb_per;     // 64-row reduction blocks per split
  size_t ws_bytes;    // fp32 partials (0 when splits == 1)
};
WPlan w_plan(int64_t M, int64_t K, int64_t N, int num_sms);
int device_sm_count();

cudaError_t launch_x_gemm(const uint16_t* dg, const uint16_t* dfc, const uint16_t* w_g, const uint16_t* w_fc,
                          uint16_t* dx, int64_t M, int64_t K, int64_t N, cudaStream_t stream);
// forward: g = x W_g + b_g, fc = x W_fc + b_fc, y = SiLU(g) fc (b_g, b_fc may be null);
// persistent tcgen05 GEMM (fwd_tc.cu)
cudaError_t launch_fwd_gemm(const uint16_t* x, const uint16_t* w_g, const uint16_t* w_fc, const uint16_t* b_g,
                            const uint16_t* b_fc, uint16_t* g, uint16_t* fc, uint16_t* y, int64_t M, int64_t K,
                            int64_t N, cudaStream_t stream);
cudaError_t launch_w_gemm(const uint16_t* x, const uint16_t* dg, const uint16_t* dfc, uint16_t* dw_g,
                          uint16_t* dw_fc, int64_t M, int64_t K, int64_t N, void* ws, const WPlan& plan,
                          cudaStream_t stream, bool accumulate = false);

// ---- GroupNorm backward (group_norm_bwd.cu); dtype 0 = f32, 1 = f16, 2 = bf16
struct GnPlan {
  int S;          // CTAs (one cluster) per (sample, group), 1..8
  int64_t slice;  // group elements per CTA (multiple of 8)
  int64_t stage;  // shared-memory stage per tensor, elements
};
GnPlan gn_plan(int64_t N, int64_t C, int64_t HxW, int64_t G, int elem_bytes, int num_sms);
// persistent double-buffered form (16-byte aligned groups); S = 0 when two buffers do not fit
GnPlan gn_pipe_plan(int64_t N, int64_t C, int64_t HxW, int64_t G, int elem_bytes, int num_sms);
// workspace for dgamma / dbeta: per-(sample, group) statistics + per-channel partials
size_t gn_workspace_bytes(int64_t N, int64_t C, int64_t G);
// dx always; dgamma, dbeta when non-null (then ws holds gn_workspace_bytes); gamma null = ones
cudaError_t launch_group_norm_bwd(const void* dy, const void* x, const void* gamma, void* dx, void* dgamma,
                                  void* dbeta, int64_t N, int64_t C, int64_t HxW, int64_t G, float eps, int dtype,
                                  void* ws, cudaStream_t stream);

// one-shot fault injection for tests of the timeout path (swg_inject_stall): the next
// launch of `kernel` (1 = x GEMM, 2 = fused x) stops issuing operand copies at ring
// entry `stall_at` and gives every pipeline wait `wait_limit` cycles. take_injection
// returns the values for that launch (stall_at -1 and the normal limit when none is armed)
// and disarms it.
struct Injection {
  int64_t stall_at;
  long long wait_limit;
};
void arm_injection(int kernel, int64_t stall_at, long long wait_limit);
Injection take_injection(int kernel);

// module status word (timeouts)
cudaError_t read_and_clear_status(uint32_t* out, cudaStream_t stream);
// device address of the status word on the current device (for kernels in other files)
uint32_t* status_word_ptr();

// ---- fused variant: b-stage math in the GEMM operand producer
struct FwPlan {
  int64_t splits, kb_per;
  size_t ws_bytes;
};
// ws_bytes = split-M dw partials (when splits > 1) + db partials [splits][2N], 256-B aligned parts
FwPlan fw_plan(int64_t M, int64_t K, int64_t N, int num_sms);
// dx (and optionally dg, dfc) from dy, g, fc, W: the work tiles [tile_begin, tile_end) (tile t = m rows
// 128 (t / tk) onwards at K block t % tk, tk = ceil(K / 512); tile_end < 0: to the last one) on one
// persistent wave of at most max_ctas CTAs (0: as many as fit)
cudaError_t launch_fused_x(const uint16_t* dy, const uint16_t* g, const uint16_t* fc, const uint16_t* w_g,
                           const uint16_t* w_fc, uint16_t* dx, uint16_t* dg, uint16_t* dfc, int64_t M, int64_t K,
                           int64_t N, cudaStream_t stream, int64_t tile_begin = 0, int64_t tile_end = -1,
                           int max_ctas = 0);
int64_t fused_x_tiles(int64_t M, int64_t K);
// CTAs of one fused w-stage launch under a plan
int64_t fused_w_ctas(int64_t K, int64_t N, const FwPlan& plan);
// dw and db from x, dy, g, fc; ws holds the split-M dw partials, then the db partials
cudaError_t launch_fused_w(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                           uint16_t* dw_g, uint16_t* dw_fc, uint16_t* db_g, uint16_t* db_fc, int64_t M, int64_t K,
                           int64_t N, void* ws, const FwPlan& plan, cudaStream_t stream, bool accumulate = false);
// the same in two parts, for a caller that runs the reduction on another stream: the kernel (dw, db
// partials into ws; with one split it writes dw itself), then the reduction of ws into dw, db.
// beside_ctas > 0 caps the reduction at that many 64-thread blocks that each fit beside a CTA of the
// fused x stage (0: the grid of the one-stream form)
cudaError_t launch_fused_w_kernel(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                                  uint16_t* dw_g, uint16_t* dw_fc, int64_t M, int64_t K, int64_t N, void* ws,
                                  const FwPlan& plan, cudaStream_t stream, bool accumulate);
cudaError_t launch_fused_w_reduce(void* ws, const FwPlan& plan, int64_t K, int64_t N, uint16_t* dw_g,
                                  uint16_t* dw_fc, uint16_t* db_g, uint16_t* db_fc, cudaStream_t stream,
                                  bool accumulate, int beside_ctas);
cudaError_t launch_w_split_reduce(const float* ws, int64_t splits, int64_t K, int64_t N, uint16_t* dw_g,
                                  uint16_t* dw_fc, cudaStream_t stream, bool accumulate = false);
// the fused w stage's kernel alone (plan.splits >= 2): fp32 partials into dw_part [splits][2][K][N] and
// db_part [splits][2N], no reduction (the caller reduces several such blocks at once)
cudaError_t launch_fused_w_partials(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                                    int64_t M, int64_t K, int64_t N, float* dw_part, float* db_part,
                                    const FwPlan& plan, cudaStream_t stream);

// tensor-map encoding (driver entry point resolved once)
bool encode_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_outer, int swizzle_bytes = 128);

}  // namespace swg
