// C ABI of the library (declared in include/swiglu_bwd.h): argument checks,
// workspace layout and kernel dispatch. No device memory is allocated here.
//
// Error model after the two-phase aclnn interface described in "SwishGrad in
// CANN ops-nn: principle, implementation and the aclnnSwishBackward guide",
// section 3.3 (null pointer -> its own code; unsupported dtype, mismatched
// dtype or shape -> invalid parameter) and section 3.5 (empty tensors
// short-circuit with no launch; a missing beta means 1.0).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "../../include/swiglu_bwd.h"
#include "swg_launch.h"

namespace {

using swg::WPlan;

constexpr int64_t kMaxDim = 0x7fffffffLL;  // TMA coordinates are 32-bit

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
inline Range rng(const void* p, int64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + static_cast<uintptr_t>(bytes)};
}
inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// true if any output range overlaps another output or any input range
bool any_overlap(const Range* outs, int nout, const Range* ins, int nin) {
  for (int i = 0; i < nout; ++i) {
    for (int j = i + 1; j < nout; ++j)
      if (overlap(outs[i], outs[j])) return true;
    for (int j = 0; j < nin; ++j)
      if (overlap(outs[i], ins[j])) return true;
  }
  return false;
}

// current device must be sm_103 (the kernels are built for sm_103a only)
swg_status check_device() {
  static std::mutex mu;
  static int known[64] = {0};  // 0 unknown, 1 ok, 2 not ok
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWG_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SWG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(mu);
  if (known[dev] == 0) {
    int maj = 0, min = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SWG_ERR_CUDA;
    known[dev] = (maj == 10 && min == 3) ? 1 : 2;
  }
  return known[dev] == 1 ? SWG_OK : SWG_ERR_UNSUPPORTED;
}

inline swg_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SWG_OK : SWG_ERR_CUDA; }

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

swg_status check_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K < 0 || N < 0) return SWG_ERR_PARAM_INVALID;
  if (M > kMaxDim || K > kMaxDim || N > kMaxDim) return SWG_ERR_UNSUPPORTED;
  if ((K % 8) != 0 || (N % 8) != 0) return SWG_ERR_UNSUPPORTED;
  return SWG_OK;
}

// zero-fill a bf16 buffer of n elements (used for sums over zero rows)
swg_status zero_bf16(void* p, int64_t n, cudaStream_t st) {
  if (n <= 0) return SWG_OK;
  return cuda_status(cudaMemsetAsync(p, 0, static_cast<size_t>(n) * 2, st));
}

}  // namespace

extern "C" {

const char* swg_status_string(swg_status s) {
  switch (s) {
    case SWG_OK: return "SWG_OK";
    case SWG_ERR_NULLPTR: return "SWG_ERR_NULLPTR: a required pointer is NULL";
    case SWG_ERR_PARAM_INVALID: return "SWG_ERR_PARAM_INVALID: invalid dtype, size or overlapping buffers";
    case SWG_ERR_UNSUPPORTED:
      return "SWG_ERR_UNSUPPORTED: K/N not a multiple of 8, misaligned pointer or device is not sm_103";
    case SWG_ERR_WORKSPACE: return "SWG_ERR_WORKSPACE: workspace missing or smaller than the query";
    case SWG_ERR_CUDA: return "SWG_ERR_CUDA: a CUDA call or kernel launch failed";
    case SWG_ERR_TIMEOUT: return "SWG_ERR_TIMEOUT: a kernel gave up waiting on a pipeline barrier";
  }
  return "SWG_ERR_?: unknown status";
}

swg_status swg_inject_stall(swg_inject_kernel kernel, int64_t entry, int64_t wait_limit_cycles) {
  if (kernel == SWG_INJECT_NONE) {
    swg::arm_injection(0, -1, 0);
    return SWG_OK;
  }
  if (kernel != SWG_INJECT_X_GEMM && kernel != SWG_INJECT_FUSED_X && kernel != SWG_INJECT_FUSED_W &&
      kernel != SWG_INJECT_FWD)
    return SWG_ERR_PARAM_INVALID;
  if (entry < 0 || wait_limit_cycles < 1024) return SWG_ERR_PARAM_INVALID;
  swg::arm_injection(static_cast<int>(kernel), entry, static_cast<long long>(wait_limit_cycles));
  return SWG_OK;
}

swg_status swg_check(swg_stream_t stream) {
  uint32_t v = 0;
  cudaError_t e = swg::read_and_clear_status(&v, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return SWG_ERR_CUDA;
  return v != 0 ? SWG_ERR_TIMEOUT : SWG_OK;
}

// ---------------------------------------------------------------- SwishGrad
// shared argument checks of the element-wise gradients (swish_grad, act_grad)
swg_status check_elementwise(const void* grad, const void* x, void* grad_x, int64_t n, swg_dtype dtype) {
  if (n < 0 || (dtype != SWG_F32 && dtype != SWG_F16 && dtype != SWG_BF16)) return SWG_ERR_PARAM_INVALID;
  if (n == 0) return SWG_OK;  // empty tensors may carry NULL data pointers
  if (grad == nullptr || x == nullptr || grad_x == nullptr) return SWG_ERR_NULLPTR;
  const int64_t es = dtype == SWG_F32 ? 4 : 2;
  const uintptr_t mask = static_cast<uintptr_t>(es - 1);
  if ((reinterpret_cast<uintptr_t>(grad) & mask) || (reinterpret_cast<uintptr_t>(x) & mask) ||
      (reinterpret_cast<uintptr_t>(grad_x) & mask))
    return SWG_ERR_UNSUPPORTED;
  // grad_x may alias grad or x exactly, but must not partially overlap either
  const Range o = rng(grad_x, n * es), a = rng(grad, n * es), b = rng(x, n * es);
  if ((overlap(o, a) && o.lo != a.lo) || (overlap(o, b) && o.lo != b.lo)) return SWG_ERR_PARAM_INVALID;
  return SWG_OK;
}

swg_status act_grad(const void* grad, const void* x, swg_act act, void* grad_x, int64_t n, swg_dtype dtype,
                    swg_stream_t stream) {
  if (act != SWG_ACT_SILU && act != SWG_ACT_GELU && act != SWG_ACT_HARDSWISH) return SWG_ERR_PARAM_INVALID;
  swg_status st = check_elementwise(grad, x, grad_x, n, dtype);
  if (st != SWG_OK || n == 0) return st;
  st = check_device();
  if (st != SWG_OK) return st;
  return cuda_status(swg::launch_act_grad(grad, x, static_cast<int>(act), grad_x, n, static_cast<int>(dtype),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- GroupNorm backward
size_t group_norm_bwd_workspace_size(int64_t N, int64_t C, int64_t HxW, int64_t G) {
  if (N <= 0 || C <= 0 || HxW <= 0 || G <= 0 || C % G != 0) return 0;
  return swg::gn_workspace_bytes(N, C, G);
}

swg_status group_norm_bwd(const void* dy, const void* x, const void* gamma, void* dx, void* dgamma, void* dbeta,
                          int64_t N, int64_t C, int64_t HxW, int64_t G, float eps, swg_dtype dtype,
                          void* workspace, size_t workspace_bytes, swg_stream_t stream) {
  if (dtype != SWG_F32 && dtype != SWG_F16 && dtype != SWG_BF16) return SWG_ERR_PARAM_INVALID;
  if (N < 0 || C < 0 || HxW < 0 || G < 1 || C % G != 0 || !(eps >= 0.0f)) return SWG_ERR_PARAM_INVALID;
  // sizes: every index fits 64 bits (N C HxW elements, and their bytes, below 2^60); the grid of
  // N G clusters of up to 8 CTAs stays below 2^31 blocks
  if (N > kMaxDim || C > kMaxDim || HxW > (int64_t(1) << 40) || N * G >= (int64_t(1) << 28))
    return SWG_ERR_UNSUPPORTED;
  if (N > 0 && C > 0 && HxW > ((int64_t(1) << 60) / N) / C) return SWG_ERR_UNSUPPORTED;
  const int64_t es = dtype == SWG_F32 ? 4 : 2;
  const int64_t n = N * C * HxW;
  const bool params = dgamma != nullptr || dbeta != nullptr;
  const uintptr_t mask = static_cast<uintptr_t>(es - 1);
  auto misaligned = [&](const void* p) { return (reinterpret_cast<uintptr_t>(p) & mask) != 0; };
  if (misaligned(dy) || misaligned(x) || misaligned(gamma) || misaligned(dx) || misaligned(dgamma) ||
      misaligned(dbeta))
    return SWG_ERR_UNSUPPORTED;
  if (n > 0 && (dy == nullptr || x == nullptr || dx == nullptr)) return SWG_ERR_NULLPTR;
  const Range outs[3] = {rng(dx, n * es), rng(dgamma, dgamma ? C * es : 0), rng(dbeta, dbeta ? C * es : 0)};
  const Range ins[3] = {rng(dy, n * es), rng(x, n * es), rng(gamma, gamma ? C * es : 0)};
  if (any_overlap(outs, 3, ins, 3)) return SWG_ERR_PARAM_INVALID;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n == 0) {
    if (C == 0 || !params) return SWG_OK;
    swg_status s = check_device();
    if (s != SWG_OK) return s;
    if (dgamma != nullptr && cudaMemsetAsync(dgamma, 0, static_cast<size_t>(C * es), st) != cudaSuccess)
      return SWG_ERR_CUDA;
    if (dbeta != nullptr && cudaMemsetAsync(dbeta, 0, static_cast<size_t>(C * es), st) != cudaSuccess)
      return SWG_ERR_CUDA;
    return SWG_OK;
  }
  if (params && (workspace == nullptr || !aligned16(workspace) ||
                 workspace_bytes < swg::gn_workspace_bytes(N, C, G)))
    return SWG_ERR_WORKSPACE;
  swg_status s = check_device();
  if (s != SWG_OK) return s;
  return cuda_status(swg::launch_group_norm_bwd(dy, x, gamma, dx, dgamma, dbeta, N, C, HxW, G, eps,
                                                static_cast<int>(dtype), params ? workspace : nullptr, st));
}

swg_status swish_grad(const void* grad, const void* x, const float* scale, void* grad_x, int64_t n,
                      swg_dtype dtype, swg_stream_t stream) {
  swg_status st = check_elementwise(grad, x, grad_x, n, dtype);
  if (st != SWG_OK || n == 0) return st;
  st = check_device();
  if (st != SWG_OK) return st;
  const float beta = scale != nullptr ? *scale : 1.0f;
  return cuda_status(swg::launch_swish_grad(grad, x, beta, grad_x, n, static_cast<int>(dtype),
                                            reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- b stage
size_t swiglu_bwd_b_workspace_size(int64_t M, int64_t N) {
  if (M <= 0 || N <= 0) return 0;
  return swg::b_workspace_bytes(M, N);
}

swg_status swiglu_bwd_b(const void* dy, const void* g, const void* fc, void* dg, void* dfc, void* db_g,
                        void* db_fc, int64_t M, int64_t N, void* workspace, size_t workspace_bytes,
                        swg_stream_t stream) {
  swg_status st = check_shape(M, 8, N);
  if (st != SWG_OK) return st;
  if (N == 0) return SWG_OK;
  // [M,N] tensors may be NULL when M == 0 (empty); [1,N] outputs are required
  if (!db_g || !db_fc || (M > 0 && (!dy || !g || !fc || !dg || !dfc))) return SWG_ERR_NULLPTR;
  const void* all[] = {dy, g, fc, dg, dfc, db_g, db_fc};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const int64_t mn = M * N * 2;
  const Range outs[] = {rng(dg, mn), rng(dfc, mn), rng(db_g, N * 2), rng(db_fc, N * 2)};
  const Range ins[] = {rng(dy, mn), rng(g, mn), rng(fc, mn)};
  if (any_overlap(outs, 4, ins, 3)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    st = zero_bf16(db_g, N, s);
    return st != SWG_OK ? st : zero_bf16(db_fc, N, s);
  }
  const size_t need = swg::b_workspace_bytes(M, N);
  if (workspace == nullptr || workspace_bytes < need) return SWG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SWG_ERR_UNSUPPORTED;
  const Range w = rng(workspace, static_cast<int64_t>(need));
  if (any_overlap(&w, 1, outs, 4) || any_overlap(&w, 1, ins, 3)) return SWG_ERR_PARAM_INVALID;
  return cuda_status(swg::launch_b_stage(
      static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(fc),
      static_cast<uint16_t*>(dg), static_cast<uint16_t*>(dfc), static_cast<uint16_t*>(db_g),
      static_cast<uint16_t*>(db_fc), M, N, workspace, s));
}

// ---------------------------------------------------------------- w stage
size_t swiglu_bwd_w_workspace_size(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  return swg::w_plan(M, K, N, swg::device_sm_count()).ws_bytes;
}

swg_status swiglu_bwd_w(const void* x, const void* dg, const void* dfc, void* dw_g, void* dw_fc, int64_t M,
                        int64_t K, int64_t N, void* workspace, size_t workspace_bytes, swg_stream_t stream) {
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (K == 0 || N == 0) return SWG_OK;
  if (!dw_g || !dw_fc || (M > 0 && (!x || !dg || !dfc))) return SWG_ERR_NULLPTR;
  const void* all[] = {x, dg, dfc, dw_g, dw_fc};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const Range outs[] = {rng(dw_g, K * N * 2), rng(dw_fc, K * N * 2)};
  const Range ins[] = {rng(x, M * K * 2), rng(dg, M * N * 2), rng(dfc, M * N * 2)};
  if (any_overlap(outs, 2, ins, 3)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    st = zero_bf16(dw_g, K * N, s);
    return st != SWG_OK ? st : zero_bf16(dw_fc, K * N, s);
  }
  const WPlan plan = swg::w_plan(M, K, N, swg::device_sm_count());
  if (plan.ws_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < plan.ws_bytes) return SWG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SWG_ERR_UNSUPPORTED;
    const Range w = rng(workspace, static_cast<int64_t>(plan.ws_bytes));
    if (any_overlap(&w, 1, outs, 2) || any_overlap(&w, 1, ins, 3)) return SWG_ERR_PARAM_INVALID;
  }
  return cuda_status(swg::launch_w_gemm(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(dg),
                                        static_cast<const uint16_t*>(dfc), static_cast<uint16_t*>(dw_g),
                                        static_cast<uint16_t*>(dw_fc), M, K, N, workspace, plan, s));
}

// ---------------------------------------------------------------- x stage
swg_status swiglu_bwd_x(const void* dg, const void* dfc, const void* w_g, const void* w_fc, void* dx, int64_t M,
                        int64_t K, int64_t N, swg_stream_t stream) {
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (M == 0 || K == 0) return SWG_OK;
  if (!dg || !dfc || !w_g || !w_fc || !dx) return SWG_ERR_NULLPTR;
  const void* all[] = {dg, dfc, w_g, w_fc, dx};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const Range outs[] = {rng(dx, M * K * 2)};
  const Range ins[] = {rng(dg, M * N * 2), rng(dfc, M * N * 2), rng(w_g, K * N * 2), rng(w_fc, K * N * 2)};
  if (any_overlap(outs, 1, ins, 4)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0) return cuda_status(cudaMemsetAsync(dx, 0, static_cast<size_t>(M * K * 2), s));
  return cuda_status(swg::launch_x_gemm(static_cast<const uint16_t*>(dg), static_cast<const uint16_t*>(dfc),
                                        static_cast<const uint16_t*>(w_g), static_cast<const uint16_t*>(w_fc),
                                        static_cast<uint16_t*>(dx), M, K, N, s));
}

// ---------------------------------------------------------------- forward
swg_status swiglu_fwd(const void* x, const void* w_g, const void* w_fc, const void* b_g, const void* b_fc, void* g,
                      void* fc, void* y, int64_t M, int64_t K, int64_t N, swg_stream_t stream) {
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (K == 0) return SWG_ERR_UNSUPPORTED;  // the products need a reduction of positive length
  if (M == 0 || N == 0) return SWG_OK;
  if (!x || !w_g || !w_fc || !g || !fc || !y) return SWG_ERR_NULLPTR;
  const void* all[] = {x, w_g, w_fc, b_g, b_fc, g, fc, y};  // null biases count as aligned
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const int64_t mn = M * N * 2, kn = K * N * 2;
  const Range outs[] = {rng(g, mn), rng(fc, mn), rng(y, mn)};
  const Range ins[] = {rng(x, M * K * 2), rng(w_g, kn), rng(w_fc, kn), rng(b_g, b_g ? N * 2 : 0),
                       rng(b_fc, b_fc ? N * 2 : 0)};
  if (any_overlap(outs, 3, ins, 5)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(swg::launch_fwd_gemm(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(w_g), static_cast<const uint16_t*>(w_fc),
      static_cast<const uint16_t*>(b_g), static_cast<const uint16_t*>(b_fc), static_cast<uint16_t*>(g),
      static_cast<uint16_t*>(fc), static_cast<uint16_t*>(y), M, K, N, s));
}

// ---------------------------------------------------------------- fused stages
swg_status swiglu_bwd_x_fused(const void* dy, const void* g, const void* fc, const void* w_g, const void* w_fc,
                              void* dx, void* dg, void* dfc, int64_t M, int64_t K, int64_t N, swg_stream_t stream) {
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (M == 0 || K == 0) return SWG_OK;
  if (!dy || !g || !fc || !w_g || !w_fc || !dx) return SWG_ERR_NULLPTR;
  if ((dg == nullptr) != (dfc == nullptr)) return SWG_ERR_NULLPTR;
  const void* all[] = {dy, g, fc, w_g, w_fc, dx, dg, dfc};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const int64_t mn = M * N * 2, kn = K * N * 2;
  const Range outs[] = {rng(dx, M * K * 2), rng(dg, dg ? mn : 0), rng(dfc, dfc ? mn : 0)};
  const Range ins[] = {rng(dy, mn), rng(g, mn), rng(fc, mn), rng(w_g, kn), rng(w_fc, kn)};
  if (any_overlap(outs, 3, ins, 5)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0) return cuda_status(cudaMemsetAsync(dx, 0, static_cast<size_t>(M * K * 2), s));
  return cuda_status(swg::launch_fused_x(
      static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(fc),
      static_cast<const uint16_t*>(w_g), static_cast<const uint16_t*>(w_fc), static_cast<uint16_t*>(dx),
      static_cast<uint16_t*>(dg), static_cast<uint16_t*>(dfc), M, K, N, s));
}

size_t swiglu_bwd_w_fused_workspace_size(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  return swg::fw_plan(M, K, N, swg::device_sm_count()).ws_bytes;
}

swg_status swiglu_bwd_w_fused(const void* x, const void* dy, const void* g, const void* fc, void* dw_g,
                              void* dw_fc, void* db_g, void* db_fc, int64_t M, int64_t K, int64_t N, void* workspace,
                              size_t workspace_bytes, swg_stream_t stream) {
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (K == 0 || N == 0) return SWG_OK;
  if (!dw_g || !dw_fc || !db_g || !db_fc || (M > 0 && (!x || !dy || !g || !fc))) return SWG_ERR_NULLPTR;
  const void* all[] = {x, dy, g, fc, dw_g, dw_fc, db_g, db_fc};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const int64_t mn = M * N * 2, kn = K * N * 2;
  const Range outs[] = {rng(dw_g, kn), rng(dw_fc, kn), rng(db_g, N * 2), rng(db_fc, N * 2)};
  const Range ins[] = {rng(x, M * K * 2), rng(dy, mn), rng(g, mn), rng(fc, mn)};
  if (any_overlap(outs, 4, ins, 4)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    st = zero_bf16(dw_g, K * N, s);
    if (st == SWG_OK) st = zero_bf16(dw_fc, K * N, s);
    if (st == SWG_OK) st = zero_bf16(db_g, N, s);
    return st != SWG_OK ? st : zero_bf16(db_fc, N, s);
  }
  const swg::FwPlan plan = swg::fw_plan(M, K, N, swg::device_sm_count());
  if (workspace == nullptr || workspace_bytes < plan.ws_bytes) return SWG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SWG_ERR_UNSUPPORTED;
  const Range w = rng(workspace, static_cast<int64_t>(plan.ws_bytes));
  if (any_overlap(&w, 1, outs, 4) || any_overlap(&w, 1, ins, 4)) return SWG_ERR_PARAM_INVALID;
  return cuda_status(swg::launch_fused_w(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(g),
      static_cast<const uint16_t*>(fc), static_cast<uint16_t*>(dw_g), static_cast<uint16_t*>(dw_fc),
      static_cast<uint16_t*>(db_g), static_cast<uint16_t*>(db_fc), M, K, N, workspace, plan, s));
}

// ---------------------------------------------------------------- whole backward from host buffers
// The fused backward with every tensor in host memory. M is cut into chunks
// (equal ones, then a short last one); while chunk c is computed (dx, and the fused w
// stage's fp32 split partials into chunk c's own slots), chunk c + 1's rows are
// copied in on one internal stream and chunk c - 1's dx is copied out on
// another, each chunk's device buffers alternating between two sets. One
// fixed-order reduction over every chunk's partials gives dw and db with one
// rounding, as in the single-call backward. Workspace layout (256-byte aligned
// regions): W_g, W_fc | two input sets (x, dy, g, fc rows of a chunk) | two dx
// sets | dw_g, dw_fc, db_g, db_fc | dw partials [S total][2][K][N] fp32 |
// db partials [S total][2N] fp32 (a single chunk: the fused w stage's own
// workspace instead of the partial blocks).
namespace {

constexpr int64_t kHostChunkRows = 32768;
constexpr int64_t kMinLastRows = 16384;

struct HostPlan {
  int64_t chunks, rows;  // chunk count, rows per chunk (multiple of 64; the last may be shorter)
  int64_t splits_total;  // sum of the chunks' M-splits (chunks > 1)
  size_t off_w, off_in[2], off_dx[2], off_out, off_dwp, off_dbp, total;
};

HostPlan host_plan(int64_t M, int64_t K, int64_t N, int sms) {
  HostPlan p{};
  // floor(M / kHostChunkRows) chunks (at most 256): all but the last of one 64-row multiple, the
  // last as short as allowed (kMinLastRows to kMinLastRows + 64 (chunks - 1) rows), so that little
  // compute and dx copy-out is left after the last rows have come in. Every chunk keeps at least 16K
  // rows, so each one splits over M (its partials path needs two splits).
  p.chunks = M >= 2 * kHostChunkRows ? std::min<int64_t>(M / kHostChunkRows, 256) : (M > 0 ? 1 : 0);
  p.rows = p.chunks > 1 ? (M - kMinLastRows) / (p.chunks - 1) / 64 * 64 : (M + 63) / 64 * 64;
  size_t off = 0;
  p.off_w = off;
  off += align256(static_cast<size_t>(2 * K * N) * 2);
  const size_t in_bytes = static_cast<size_t>(p.rows) * static_cast<size_t>(K + 3 * N) * 2;
  const size_t dx_bytes = static_cast<size_t>(p.rows) * static_cast<size_t>(K) * 2;
  for (int b = 0; b < 2; ++b) {
    p.off_in[b] = off;
    off += align256(in_bytes);
  }
  for (int b = 0; b < 2; ++b) {
    p.off_dx[b] = off;
    off += align256(dx_bytes);
  }
  p.off_out = off;
  off += align256(static_cast<size_t>(2 * K * N + 2 * N) * 2);
  if (p.chunks > 1) {
    for (int64_t c = 0; c < p.chunks; ++c) {
      const int64_t r = std::min(p.rows, M - c * p.rows);
      p.splits_total += swg::fw_plan(r, K, N, sms).splits;
    }
    p.off_dwp = off;
    off += align256(static_cast<size_t>(p.splits_total) * 2 * K * N * 4);
    p.off_dbp = off;
    off += align256(static_cast<size_t>(p.splits_total) * 2 * N * 4);
  } else {
    p.off_dwp = off;
    off += align256(p.chunks == 1 ? swg::fw_plan(M, K, N, sms).ws_bytes : 0);
    p.off_dbp = p.off_dwp;
  }
  p.total = off;
  return p;
}

// the internal copy streams and the events that order them against the caller's stream (per device,
// created once; the enqueue of one call holds the lock, so calls from several host threads take turns)
struct HostStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, w_in = nullptr, reduced = nullptr, end = nullptr;
  cudaEvent_t loaded[2] = {}, computed[2] = {}, dx_out[2] = {};
};
std::mutex g_host_mu;
HostStreams g_host[64];

cudaError_t host_streams(int dev, HostStreams** out) {
  HostStreams& h = g_host[dev];
  if (h.h2d == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking);
    cudaEvent_t* evs[] = {&h.start, &h.w_in, &h.reduced, &h.end, &h.loaded[0], &h.loaded[1],
                          &h.computed[0], &h.computed[1], &h.dx_out[0], &h.dx_out[1]};
    for (cudaEvent_t* ev : evs)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  *out = &h;
  return cudaSuccess;
}

}  // namespace

size_t swiglu_bwd_host_workspace_size(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K <= 0 || N <= 0) return 0;
  return host_plan(M, K, N, swg::device_sm_count()).total;
}

swg_status swiglu_bwd_host(const void* x, const void* w_g, const void* w_fc, const void* dy, const void* g,
                           const void* fc, void* dx, void* dw_g, void* dw_fc, void* db_g, void* db_fc, int64_t M,
                           int64_t K, int64_t N, void* workspace, size_t workspace_bytes, swg_stream_t stream) {
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (K == 0 || N == 0) return SWG_OK;
  if (!w_g || !w_fc || !dw_g || !dw_fc || !db_g || !db_fc) return SWG_ERR_NULLPTR;
  if (M > 0 && (!x || !dy || !g || !fc || !dx)) return SWG_ERR_NULLPTR;
  const int64_t kn = K * N * 2, mn = M * N * 2;
  const Range outs[] = {rng(dx, M * K * 2), rng(dw_g, kn), rng(dw_fc, kn), rng(db_g, N * 2), rng(db_fc, N * 2)};
  const Range ins[] = {rng(x, M * K * 2), rng(w_g, kn), rng(w_fc, kn), rng(dy, mn), rng(g, mn), rng(fc, mn)};
  if (any_overlap(outs, 5, ins, 6)) return SWG_ERR_PARAM_INVALID;
  st = check_device();
  if (st != SWG_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWG_ERR_CUDA;
  const int sms = swg::device_sm_count();
  const HostPlan hp = host_plan(M, K, N, sms);
  if (workspace == nullptr || workspace_bytes < hp.total) return SWG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SWG_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lk(g_host_mu);
  HostStreams* hs = nullptr;
  if (host_streams(dev, &hs) != cudaSuccess) return SWG_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto dev16 = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
  uint16_t* wg_d = dev16(hp.off_w);
  uint16_t* wfc_d = wg_d + K * N;
  uint16_t* dwg_d = dev16(hp.off_out);
  uint16_t* dwfc_d = dwg_d + K * N;
  uint16_t* dbg_d = dwfc_d + K * N;
  uint16_t* dbfc_d = dbg_d + N;
  const auto* xh = static_cast<const uint8_t*>(x);
  const auto* dyh = static_cast<const uint8_t*>(dy);
  const auto* gh = static_cast<const uint8_t*>(g);
  const auto* fch = static_cast<const uint8_t*>(fc);
  auto* dxh = static_cast<uint8_t*>(dx);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };

  ok(cudaEventRecord(hs->start, cs));
  ok(cudaStreamWaitEvent(hs->h2d, hs->start, 0));
  ok(cudaStreamWaitEvent(hs->d2h, hs->start, 0));
  ok(cudaMemcpyAsync(wg_d, w_g, kn, h2d, hs->h2d));
  ok(cudaMemcpyAsync(wfc_d, w_fc, kn, h2d, hs->h2d));
  ok(cudaEventRecord(hs->w_in, hs->h2d));
  ok(cudaStreamWaitEvent(cs, hs->w_in, 0));
  if (M == 0) {
    ok(cudaMemsetAsync(dwg_d, 0, static_cast<size_t>(2 * K * N + 2 * N) * 2, cs));
  }
  int64_t split_off = 0;
  for (int64_t c = 0; c < hp.chunks && e == cudaSuccess; ++c) {
    const int b = static_cast<int>(c & 1);
    const int64_t r0 = c * hp.rows, rows = std::min(hp.rows, M - r0);
    uint16_t* xin = dev16(hp.off_in[b]);
    uint16_t* dyin = xin + hp.rows * K;
    uint16_t* gin = dyin + hp.rows * N;
    uint16_t* fcin = gin + hp.rows * N;
    uint16_t* dxo = dev16(hp.off_dx[b]);
    // rows of chunk c in; buffer set b was last read by chunk c - 2's kernels
    if (c >= 2) ok(cudaStreamWaitEvent(hs->h2d, hs->computed[b], 0));
    ok(cudaMemcpyAsync(xin, xh + r0 * K * 2, static_cast<size_t>(rows * K * 2), h2d, hs->h2d));
    ok(cudaMemcpyAsync(dyin, dyh + r0 * N * 2, static_cast<size_t>(rows * N * 2), h2d, hs->h2d));
    ok(cudaMemcpyAsync(gin, gh + r0 * N * 2, static_cast<size_t>(rows * N * 2), h2d, hs->h2d));
    ok(cudaMemcpyAsync(fcin, fch + r0 * N * 2, static_cast<size_t>(rows * N * 2), h2d, hs->h2d));
    ok(cudaEventRecord(hs->loaded[b], hs->h2d));
    // compute; dx set b was last copied out for chunk c - 2
    ok(cudaStreamWaitEvent(cs, hs->loaded[b], 0));
    if (c >= 2) ok(cudaStreamWaitEvent(cs, hs->dx_out[b], 0));
    ok(swg::launch_fused_x(dyin, gin, fcin, wg_d, wfc_d, dxo, nullptr, nullptr, rows, K, N, cs));
    if (hp.chunks == 1) {
      const swg::FwPlan fp = swg::fw_plan(rows, K, N, sms);
      ok(swg::launch_fused_w(xin, dyin, gin, fcin, dwg_d, dwfc_d, dbg_d, dbfc_d, rows, K, N, ws + hp.off_dwp, fp,
                             cs));
    } else {
      const swg::FwPlan fp = swg::fw_plan(rows, K, N, sms);
      float* dwp = reinterpret_cast<float*>(ws + hp.off_dwp) + split_off * 2 * K * N;
      float* dbp = reinterpret_cast<float*>(ws + hp.off_dbp) + split_off * 2 * N;
      ok(swg::launch_fused_w_partials(xin, dyin, gin, fcin, rows, K, N, dwp, dbp, fp, cs));
      split_off += fp.splits;
    }
    ok(cudaEventRecord(hs->computed[b], cs));
    // dx of chunk c out
    ok(cudaStreamWaitEvent(hs->d2h, hs->computed[b], 0));
    ok(cudaMemcpyAsync(dxh + r0 * K * 2, dxo, static_cast<size_t>(rows * K * 2), d2h, hs->d2h));
    ok(cudaEventRecord(hs->dx_out[b], hs->d2h));
  }
  if (hp.chunks > 1) {
    ok(swg::launch_w_split_reduce(reinterpret_cast<const float*>(ws + hp.off_dwp), hp.splits_total, K, N, dwg_d,
                                  dwfc_d, cs));
    ok(swg::launch_db_reduce(reinterpret_cast<const float*>(ws + hp.off_dbp), hp.splits_total, N, dbg_d, dbfc_d,
                             cs));
  }
  ok(cudaEventRecord(hs->reduced, cs));
  ok(cudaStreamWaitEvent(hs->d2h, hs->reduced, 0));
  ok(cudaMemcpyAsync(dw_g, dwg_d, kn, d2h, hs->d2h));
  ok(cudaMemcpyAsync(dw_fc, dwfc_d, kn, d2h, hs->d2h));
  ok(cudaMemcpyAsync(db_g, dbg_d, N * 2, d2h, hs->d2h));
  ok(cudaMemcpyAsync(db_fc, dbfc_d, N * 2, d2h, hs->d2h));
  ok(cudaEventRecord(hs->end, hs->d2h));
  ok(cudaStreamWaitEvent(cs, hs->end, 0));
  return cuda_status(e);
}

// ---------------------------------------------------------------- whole backward
// Unfused workspace layout: [dg scratch 2MN | dfc scratch 2MN] (only when the
// caller passes NULL dg/dfc) | b-stage partials | w-stage partials; each
// region starts on a 256-byte boundary.
// SWG_AUTO: the chain measured faster for the shape on GB300. The fused chain
// forms dg, dfc once per 512 columns of K in each of its two kernels, the
// unfused one once in the b stage but writes and re-reads them through HBM.
// Measured (whole backward, N = 1024 unless stated): K = 512, M = 220000:
// fused 0.80 ms, unfused 1.07 ms; K = 512, M = 65537: 0.285 vs 0.346 ms;
// K = 512, M <= 4097: fused slower (fixed costs of its two persistent
// launches); K = 4096, N = 14336, M = 16384: fused 6.85 ms, unfused 5.48 ms.
namespace {

bool auto_fused(int64_t M, int64_t K) { return K <= 512 && M >= 32768; }

unsigned resolve_auto(int64_t M, int64_t K, unsigned flags) {
  if (!(flags & SWG_AUTO)) return flags;
  flags &= ~(SWG_AUTO | SWG_FUSED);
  return auto_fused(M, K) ? (flags | SWG_FUSED) : flags;
}

// The fused chain's x-stage work split: when the w stage occupies fewer CTAs than the GPU has
// SMs, the x stage's last side_tiles tiles run on side_ctas CTAs beside the w stage and the
// other main_tiles tiles in one persistent wave after it. The side share is what makes the
// main part one wave round shorter (main_tiles = (rounds - 1) * SMs), and it is taken only when
// its own rounds fit well inside the w stage. By operand volume a w-stage CTA does the work of
// kb_per / (2 * ceil(N / 64)) x-stage tiles (a 64-row stage of one band against a 128-row tile
// over all bands); in time it takes about three quarters of that (measured at K = 512,
// N = 1024: 382 stages against 8.8 tiles). The side rounds may use 0.6 of the volume figure,
// about 80% of the w stage's time.
struct FxSplit {
  int64_t main_tiles = 0, side_tiles = 0;
  int side_ctas = 0;
};
FxSplit fx_split(int64_t M, int64_t K, int64_t N, const swg::FwPlan& plan, int sms) {
  FxSplit sp;
  const int64_t tiles = swg::fused_x_tiles(M, K);
  sp.main_tiles = tiles;
  const int64_t idle = sms - swg::fused_w_ctas(K, N, plan);
  const int64_t rounds = (tiles + sms - 1) / sms;
  if (idle <= 0 || rounds < 2) return sp;
  const int64_t main = (rounds - 1) * sms, side = tiles - main;
  const int64_t side_rounds = (side + idle - 1) / idle;
  const int64_t nst = (N + 63) / 64;
  if (side_rounds * 2 * nst * 5 > plan.kb_per * 3) return sp;
  sp.main_tiles = main;
  sp.side_tiles = side;
  sp.side_ctas = static_cast<int>(idle);
  return sp;
}

// the side stream of the fused chain and its fork / join events (per device, created once;
// the enqueue of one call holds the lock)
struct SideStream {
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, fw_done = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[64];

cudaError_t side_stream(int dev, SideStream** out) {
  SideStream& h = g_side[dev];
  if (h.side == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&h.side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.join, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.fw_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  *out = &h;
  return cudaSuccess;
}

}  // namespace

size_t swiglu_bwd_workspace_size(int64_t M, int64_t K, int64_t N, unsigned flags) {
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  flags = resolve_auto(M, K, flags);
  const bool fused = (flags & SWG_FUSED) != 0;
  if (fused) return swg::fw_plan(M, K, N, swg::device_sm_count()).ws_bytes;
  size_t total = 0;
  if (!(flags & SWG_WS_DG_GIVEN)) total += 2 * align256(static_cast<size_t>(M) * N * 2);
  total += align256(swg::b_workspace_bytes(M, N));
  total += align256(swg::w_plan(M, K, N, swg::device_sm_count()).ws_bytes);
  return total;
}

int swiglu_bwd_kernel_count(int64_t M, int64_t K, int64_t N, unsigned flags) {
  if ((flags & ~(SWG_FUSED | SWG_ACCUMULATE | SWG_WS_DG_GIVEN | SWG_AUTO)) != 0) return 0;
  if (check_shape(M, K, N) != SWG_OK || M <= 0 || K == 0 || N == 0) return 0;
  flags = resolve_auto(M, K, flags);
  const int sms = swg::device_sm_count();
  if (flags & SWG_FUSED) {
    const swg::FwPlan fplan = swg::fw_plan(M, K, N, sms);
    const FxSplit sp = fx_split(M, K, N, fplan, sms);
    // x stage (one or two launches), w stage, its dw and db reductions (one launch)
    return (sp.side_tiles > 0 ? 2 : 1) + 1 + 1;
  }
  // b stage and its db reduce, w GEMM and its split reduce, x GEMM
  return 2 + 1 + (swg::w_plan(M, K, N, sms).splits > 1 ? 1 : 0) + 1;
}

swg_status swiglu_bwd(const void* x, const void* w_g, const void* w_fc, const void* dy, const void* g,
                      const void* fc, void* dg, void* dfc, void* dx, void* dw_g, void* dw_fc, void* db_g,
                      void* db_fc, int64_t M, int64_t K, int64_t N, unsigned flags, void* workspace,
                      size_t workspace_bytes, swg_stream_t stream) {
  if ((flags & ~(SWG_FUSED | SWG_ACCUMULATE | SWG_WS_DG_GIVEN | SWG_AUTO)) != 0) return SWG_ERR_PARAM_INVALID;
  flags = resolve_auto(M, K, flags);
  const bool acc = (flags & SWG_ACCUMULATE) != 0;
  swg_status st = check_shape(M, K, N);
  if (st != SWG_OK) return st;
  if (K == 0 || N == 0) return SWG_OK;
  // tensors with an M dimension may be NULL when M == 0 (empty)
  if (!w_g || !w_fc || !dw_g || !dw_fc || !db_g || !db_fc) return SWG_ERR_NULLPTR;
  if (M > 0 && (!x || !dy || !g || !fc || !dx)) return SWG_ERR_NULLPTR;
  if (M > 0 && (dg == nullptr) != (dfc == nullptr)) return SWG_ERR_NULLPTR;
  if (M == 0) dg = dfc = nullptr;
  const void* all[] = {x, w_g, w_fc, dy, g, fc, dx, dw_g, dw_fc, db_g, db_fc};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  if (dg != nullptr && (!aligned16(dg) || !aligned16(dfc))) return SWG_ERR_UNSUPPORTED;
  const int64_t mn = M * N * 2, kn = K * N * 2;
  const Range outs[] = {rng(dx, M * K * 2), rng(dw_g, kn), rng(dw_fc, kn), rng(db_g, N * 2), rng(db_fc, N * 2),
                        rng(dg, dg ? mn : 0), rng(dfc, dfc ? mn : 0)};
  const Range ins[] = {rng(x, M * K * 2), rng(w_g, kn), rng(w_fc, kn), rng(dy, mn), rng(g, mn), rng(fc, mn)};
  if (any_overlap(outs, 7, ins, 6)) return SWG_ERR_PARAM_INVALID;
  if (M == 0 && acc) return SWG_OK;  // a sum over no rows adds nothing: no work at all
  st = check_device();
  if (st != SWG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    st = zero_bf16(dw_g, K * N, s);
    if (st == SWG_OK) st = zero_bf16(dw_fc, K * N, s);
    if (st == SWG_OK) st = zero_bf16(db_g, N, s);
    if (st == SWG_OK) st = zero_bf16(db_fc, N, s);
    return st;
  }
  const unsigned wsflags = flags | (dg != nullptr ? SWG_WS_DG_GIVEN : 0u);
  const size_t need = swiglu_bwd_workspace_size(M, K, N, wsflags);
  if (workspace == nullptr || workspace_bytes < need) return SWG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return SWG_ERR_UNSUPPORTED;
  const Range w = rng(workspace, static_cast<int64_t>(need));
  if (any_overlap(&w, 1, outs, 7) || any_overlap(&w, 1, ins, 6)) return SWG_ERR_PARAM_INVALID;

  uint8_t* wp = static_cast<uint8_t*>(workspace);
  if (flags & SWG_FUSED) {
    const int sms = swg::device_sm_count();
    const swg::FwPlan fplan = swg::fw_plan(M, K, N, sms);
    const FxSplit sp = fx_split(M, K, N, fplan, sms);
    auto fx = [&](cudaStream_t cs, int64_t t0, int64_t t1, int ctas) {
      return swg::launch_fused_x(static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(g),
                                 static_cast<const uint16_t*>(fc), static_cast<const uint16_t*>(w_g),
                                 static_cast<const uint16_t*>(w_fc), static_cast<uint16_t*>(dx),
                                 static_cast<uint16_t*>(dg), static_cast<uint16_t*>(dfc), M, K, N, cs, t0, t1, ctas);
    };
    auto fw = [&]() {
      return swg::launch_fused_w(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(dy),
                                 static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(fc),
                                 static_cast<uint16_t*>(dw_g), static_cast<uint16_t*>(dw_fc),
                                 static_cast<uint16_t*>(db_g), static_cast<uint16_t*>(db_fc), M, K, N, wp, fplan,
                                 s, acc);
    };
    if (sp.side_tiles == 0) {
      cudaError_t e = fx(s, 0, -1, 0);
      if (e == cudaSuccess) e = fw();
      return cuda_status(e);
    }
    // the w stage leaves SMs free: the last x-stage tiles run there at the same time, on a
    // side stream ordered after everything before this call, and the caller's stream waits
    // for them at the end; the other x-stage tiles follow the w stage in one persistent wave
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SWG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_side_mu);
    SideStream* ss = nullptr;
    if (side_stream(dev, &ss) != cudaSuccess) return SWG_ERR_CUDA;
    cudaError_t e = cudaEventRecord(ss->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->side, ss->fork, 0);
    if (e == cudaSuccess)
      e = swg::launch_fused_w_kernel(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(dy),
                                     static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(fc),
                                     static_cast<uint16_t*>(dw_g), static_cast<uint16_t*>(dw_fc), M, K, N, wp, fplan,
                                     s, acc);
    if (e == cudaSuccess) e = cudaEventRecord(ss->fw_done, s);
    if (e == cudaSuccess) e = fx(ss->side, sp.main_tiles, sp.main_tiles + sp.side_tiles, sp.side_ctas);
    // the w stage's reduction, too, goes on the side stream, in blocks small enough to run beside the
    // x stage's persistent wave, so that it leaves the critical path
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->side, ss->fw_done, 0);
    if (e == cudaSuccess)
      e = swg::launch_fused_w_reduce(wp, fplan, K, N, static_cast<uint16_t*>(dw_g), static_cast<uint16_t*>(dw_fc),
                                     static_cast<uint16_t*>(db_g), static_cast<uint16_t*>(db_fc), ss->side, acc,
                                     sms);
    if (e == cudaSuccess) e = cudaEventRecord(ss->join, ss->side);
    if (e == cudaSuccess) e = fx(s, 0, sp.main_tiles, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ss->join, 0);
    return cuda_status(e);
  }
  uint16_t* dgp = static_cast<uint16_t*>(dg);
  uint16_t* dfcp = static_cast<uint16_t*>(dfc);
  if (dgp == nullptr) {
    dgp = reinterpret_cast<uint16_t*>(wp);
    wp += align256(static_cast<size_t>(mn));
    dfcp = reinterpret_cast<uint16_t*>(wp);
    wp += align256(static_cast<size_t>(mn));
  }
  void* bws = wp;
  wp += align256(swg::b_workspace_bytes(M, N));
  void* wws = wp;
  const WPlan plan = swg::w_plan(M, K, N, swg::device_sm_count());

  cudaError_t e = swg::launch_b_stage(static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(g),
                                      static_cast<const uint16_t*>(fc), dgp, dfcp, static_cast<uint16_t*>(db_g),
                                      static_cast<uint16_t*>(db_fc), M, N, bws, s, acc);
  if (e != cudaSuccess) return SWG_ERR_CUDA;
  e = swg::launch_w_gemm(static_cast<const uint16_t*>(x), dgp, dfcp, static_cast<uint16_t*>(dw_g),
                         static_cast<uint16_t*>(dw_fc), M, K, N, wws, plan, s, acc);
  if (e != cudaSuccess) return SWG_ERR_CUDA;
  e = swg::launch_x_gemm(dgp, dfcp, static_cast<const uint16_t*>(w_g), static_cast<const uint16_t*>(w_fc),
                         static_cast<uint16_t*>(dx), M, K, N, s);
  return cuda_status(e);
}

}  // extern "C"
