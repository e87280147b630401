// SwishGrad: grad_x = grad * sigma(beta x) * (1 + beta x (1 - sigma(beta x))).
//
// Source: "SwishGrad in CANN ops-nn: principle, implementation and the
// aclnnSwishBackward guide", section 1.2 (formula) and section 2.4 (fp16/bf16
// widened to fp32, result narrowed round-to-nearest-even; fp32 stays fp32).
//
// The same streaming kernels also run the sibling activation gradients that
// the Ascend C backward blog post names (GELU, HardSwish; SiLU is SwishGrad
// with beta = 1), each as grad_x = grad * f'(x) in fp32:
//   GELU (exact):  f'(x) = Phi(x) + x phi(x),  Phi(x) = (1 + erf(x / sqrt 2)) / 2,
//                  phi(x) = exp(-x^2 / 2) / sqrt(2 pi). erf by Abramowitz and
//                  Stegun, Handbook of Mathematical Functions, formula 7.1.26
//                  (|error| <= 1.5e-7), whose e^{-z^2} factor is phi's own
//                  exponential, so one ex2 and one rcp serve both terms
//   HardSwish:     f(x) = x min(max(x + 3, 0), 6) / 6;  f'(x) = 0 for x <= -3,
//                  x / 3 + 1/2 for -3 < x < 3, 1 for x >= 3 (kinks as PyTorch)
//
// HBM-bound: 3 * n * sizeof(T) bytes per call. The body moves 16-byte vectors
// with streaming (evict-first) loads and stores, kUnroll vectors per thread in
// flight; a scalar kernel takes the unaligned head and the ragged tail, or the
// whole array when the three pointers are misaligned relative to each other.
// The vector kernel is launched as a programmatic dependent launch: it may be
// scheduled while the previous kernel on the stream drains, waits
// (griddepcontrol.wait) until that kernel has completed and its writes are
// visible before it reads anything, and lets a following kernel that opted in
// do the same. In a stream of calls this hides the launch gap (measured on
// 2^24 bf16: 17.1 -> 16.1 us per call averaged over back-to-back calls).
#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 1;  // vectors per thread: many small CTAs measured fastest (2^24 bf16: 4% over 4)

// two elements: t = beta x, grad_x = grad * s * (1 + t (1 - s)), s = sigma(t)
__device__ __forceinline__ float2 swish_grad_f2(float2 grad, float2 x, float beta) {
  const float2 t = __fmul2_rn(make_float2(beta, beta), x);
  const Sig2 q = sigmoid_pair2(t);
  return __fmul2_rn(grad, __fmul2_rn(q.s, __ffma2_rn(t, q.sc, make_float2(1.0f, 1.0f))));
}

// one operation per kernel instance: grad_x for two elements at a time
struct OpSwish {
  float beta;
  __device__ __forceinline__ float2 f2(float2 g, float2 x) const { return swish_grad_f2(g, x, beta); }
};
__device__ __forceinline__ float gelu_d(float x) {
  // z = |x| / sqrt 2; erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^{-z^2}, t = 1 / (1 + p z)
  const float z = fabsf(x) * 0.70710678118654752f;
  const float e = ex2_approx(-(z * z) * kLog2e);  // e^{-z^2} = e^{-x^2 / 2}
  const float t = rcp_approx(fmaf(0.3275911f, z, 1.0f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f),
               0.254829592f);
  const float tail = 0.5f * poly * e;  // (1 - erf(z)) / 2
  const float cdf = x >= 0.0f ? 1.0f - tail : tail;
  return fmaf(x, 0.39894228040143268f * e, cdf);
}
struct OpGelu {
  __device__ __forceinline__ float2 f2(float2 g, float2 x) const {
    return make_float2(g.x * gelu_d(x.x), g.y * gelu_d(x.y));
  }
};
__device__ __forceinline__ float hardswish_d(float x) {
  return x <= -3.0f ? 0.0f : (x < 3.0f ? fmaf(x, 1.0f / 3.0f, 0.5f) : 1.0f);
}
struct OpHardSwish {
  __device__ __forceinline__ float2 f2(float2 g, float2 x) const {
    return make_float2(g.x * hardswish_d(x.x), g.y * hardswish_d(x.y));
  }
};

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
  static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
};
template <>
struct Elem<__half> {
  static __device__ __forceinline__ float ld(const __half* p) { return __half2float(*p); }
  static __device__ __forceinline__ void st(__half* p, float v) { *p = __float2half_rn(v); }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// one 16-byte vector: 4 fp32 or 8 fp16/bf16
template <class Op>
__device__ __forceinline__ uint4 vec_apply(uint4 g, uint4 x, const Op& op, float*) {
  const float2 a = op.f2(make_float2(__uint_as_float(g.x), __uint_as_float(g.y)),
                         make_float2(__uint_as_float(x.x), __uint_as_float(x.y)));
  const float2 b = op.f2(make_float2(__uint_as_float(g.z), __uint_as_float(g.w)),
                         make_float2(__uint_as_float(x.z), __uint_as_float(x.w)));
  return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b.x), __float_as_uint(b.y));
}
template <class Op>
__device__ __forceinline__ uint32_t pair_h(uint32_t g, uint32_t x, const Op& op) {
  const __half2 gh = *reinterpret_cast<const __half2*>(&g);
  const __half2 xh = *reinterpret_cast<const __half2*>(&x);
  const float2 r = op.f2(__half22float2(gh), __half22float2(xh));
  __half2 o = __floats2half2_rn(r.x, r.y);
  return *reinterpret_cast<uint32_t*>(&o);
}
template <class Op>
__device__ __forceinline__ uint4 vec_apply(uint4 g, uint4 x, const Op& op, __half*) {
  return make_uint4(pair_h(g.x, x.x, op), pair_h(g.y, x.y, op), pair_h(g.z, x.z, op), pair_h(g.w, x.w, op));
}
template <class Op>
__device__ __forceinline__ uint32_t pair_b(uint32_t g, uint32_t x, const Op& op) {
  const float2 r = op.f2(bf16x2_to_f2(g), bf16x2_to_f2(x));
  return pack_bf16x2(r.x, r.y);
}
template <class Op>
__device__ __forceinline__ uint4 vec_apply(uint4 g, uint4 x, const Op& op, __nv_bfloat16*) {
  return make_uint4(pair_b(g.x, x.x, op), pair_b(g.y, x.y, op), pair_b(g.z, x.z, op), pair_b(g.w, x.w, op));
}

template <typename T, class Op>
__global__ void __launch_bounds__(kThreads) swish_grad_vec_kernel(const uint4* grad, const uint4* x,
                                                                   uint4* out,
                                                                   int64_t nvec, Op op) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t base = static_cast<int64_t>(blockIdx.x) * (kThreads * kUnroll) + threadIdx.x;
  uint4 gv[kUnroll], xv[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t i = base + static_cast<int64_t>(u) * kThreads;
    if (i < nvec) {
      gv[u] = __ldcs(grad + i);
      xv[u] = __ldcs(x + i);
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t i = base + static_cast<int64_t>(u) * kThreads;
    if (i < nvec) __stcs(out + i, vec_apply(gv[u], xv[u], op, static_cast<T*>(nullptr)));
  }
}

// Elements [0, head) and [tail, n): index j < head maps to j, else to tail + (j - head).
template <typename T, class Op>
__global__ void __launch_bounds__(kThreads) swish_grad_scalar_kernel(const T* grad, const T* x, T* out,
                                                                      int64_t head, int64_t tail, int64_t n,
                                                                      Op op) {
  const int64_t count = head + (n - tail);
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < count;
       j += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t i = j < head ? j : tail + (j - head);
    Elem<T>::st(out + i, op.f2(make_float2(Elem<T>::ld(grad + i), 0.0f), make_float2(Elem<T>::ld(x + i), 0.0f)).x);
  }
}

template <typename T, class Op>
cudaError_t run(const void* grad_v, const void* x_v, const Op& op, void* out_v, int64_t n, cudaStream_t stream) {
  const T* grad = static_cast<const T*>(grad_v);
  const T* x = static_cast<const T*>(x_v);
  T* out = static_cast<T*>(out_v);
  constexpr int64_t kVec = 16 / sizeof(T);
  const uintptr_t ag = reinterpret_cast<uintptr_t>(grad) & 15u;
  const uintptr_t ax = reinterpret_cast<uintptr_t>(x) & 15u;
  const uintptr_t ao = reinterpret_cast<uintptr_t>(out) & 15u;
  int64_t head = n, tail = n, nvec = 0;
  if (ag == ax && ag == ao && (ag % sizeof(T)) == 0) {
    head = static_cast<int64_t>(((16u - ag) & 15u) / sizeof(T));
    if (head > n) head = n;
    nvec = (n - head) / kVec;
    tail = head + nvec * kVec;
  }
  if (nvec > 0) {
    const int64_t blocks = (nvec + kThreads * kUnroll - 1) / (kThreads * kUnroll);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, swish_grad_vec_kernel<T, Op>,
                                             reinterpret_cast<const uint4*>(grad + head),
                                             reinterpret_cast<const uint4*>(x + head),
                                             reinterpret_cast<uint4*>(out + head), nvec, op);
    if (e != cudaSuccess) return e;
  }
  const int64_t rest = head + (n - tail);
  if (rest > 0) {
    int64_t blocks = (rest + kThreads - 1) / kThreads;
    if (blocks > 4096) blocks = 4096;
    swish_grad_scalar_kernel<T, Op><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(grad, x, out, head,
                                                                                            tail, n, op);
  }
  return cudaGetLastError();
}

template <class Op>
cudaError_t dispatch(const void* grad, const void* x, const Op& op, void* grad_x, int64_t n, int dtype,
                     cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  switch (dtype) {
    case 0: return run<float>(grad, x, op, grad_x, n, stream);
    case 1: return run<__half>(grad, x, op, grad_x, n, stream);
    default: return run<__nv_bfloat16>(grad, x, op, grad_x, n, stream);
  }
}

}  // namespace

cudaError_t launch_swish_grad(const void* grad, const void* x, float beta, void* grad_x, int64_t n, int dtype,
                              cudaStream_t stream) {
  return dispatch(grad, x, OpSwish{beta}, grad_x, n, dtype, stream);
}

cudaError_t launch_act_grad(const void* grad, const void* x, int act, void* grad_x, int64_t n, int dtype,
                            cudaStream_t stream) {
  switch (act) {
    case 0: return dispatch(grad, x, OpSwish{1.0f}, grad_x, n, dtype, stream);  // SiLU = SwishGrad, beta 1
    case 1: return dispatch(grad, x, OpGelu{}, grad_x, n, dtype, stream);
    default: return dispatch(grad, x, OpHardSwish{}, grad_x, n, dtype, stream);
  }
}

}  // namespace swg
