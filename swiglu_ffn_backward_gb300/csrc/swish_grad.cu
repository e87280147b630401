// SwishGrad: grad_x = grad * sigma(beta x) * (1 + beta x (1 - sigma(beta x))).
//
// Source: "SwishGrad in CANN ops-nn: principle, implementation and the
// aclnnSwishBackward guide", section 1.2 (formula) and section 2.4 (fp16/bf16
// widened to fp32, result narrowed round-to-nearest-even; fp32 stays fp32).
//
// HBM-bound: 3 * n * sizeof(T) bytes per call. The body moves 16-byte vectors
// with streaming (evict-first) loads and stores, kUnroll vectors per thread in
// flight; a scalar kernel takes the unaligned head and the ragged tail, or the
// whole array when the three pointers are misaligned relative to each other.
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
__device__ __forceinline__ float swish_grad_f32(float grad, float x, float beta) {
  return swish_grad_f2(make_float2(grad, 0.0f), make_float2(x, 0.0f), beta).x;
}

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
__device__ __forceinline__ uint4 vec_apply(uint4 g, uint4 x, float beta, float*) {
  const float2 a = swish_grad_f2(make_float2(__uint_as_float(g.x), __uint_as_float(g.y)),
                                 make_float2(__uint_as_float(x.x), __uint_as_float(x.y)), beta);
  const float2 b = swish_grad_f2(make_float2(__uint_as_float(g.z), __uint_as_float(g.w)),
                                 make_float2(__uint_as_float(x.z), __uint_as_float(x.w)), beta);
  return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b.x), __float_as_uint(b.y));
}
__device__ __forceinline__ uint32_t pair_h(uint32_t g, uint32_t x, float beta) {
  const __half2 gh = *reinterpret_cast<const __half2*>(&g);
  const __half2 xh = *reinterpret_cast<const __half2*>(&x);
  const float2 r = swish_grad_f2(__half22float2(gh), __half22float2(xh), beta);
  __half2 o = __floats2half2_rn(r.x, r.y);
  return *reinterpret_cast<uint32_t*>(&o);
}
__device__ __forceinline__ uint4 vec_apply(uint4 g, uint4 x, float beta, __half*) {
  return make_uint4(pair_h(g.x, x.x, beta), pair_h(g.y, x.y, beta), pair_h(g.z, x.z, beta),
                    pair_h(g.w, x.w, beta));
}
__device__ __forceinline__ uint32_t pair_b(uint32_t g, uint32_t x, float beta) {
  const float2 r = swish_grad_f2(bf16x2_to_f2(g), bf16x2_to_f2(x), beta);
  return pack_bf16x2(r.x, r.y);
}
__device__ __forceinline__ uint4 vec_apply(uint4 g, uint4 x, float beta, __nv_bfloat16*) {
  return make_uint4(pair_b(g.x, x.x, beta), pair_b(g.y, x.y, beta), pair_b(g.z, x.z, beta),
                    pair_b(g.w, x.w, beta));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) swish_grad_vec_kernel(const uint4* grad, const uint4* x,
                                                                   uint4* out,
                                                                   int64_t nvec, float beta) {
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
    if (i < nvec) __stcs(out + i, vec_apply(gv[u], xv[u], beta, static_cast<T*>(nullptr)));
  }
}

// Elements [0, head) and [tail, n): index j < head maps to j, else to tail + (j - head).
template <typename T>
__global__ void __launch_bounds__(kThreads) swish_grad_scalar_kernel(const T* grad, const T* x, T* out,
                                                                      int64_t head, int64_t tail, int64_t n,
                                                                      float beta) {
  const int64_t count = head + (n - tail);
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < count;
       j += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t i = j < head ? j : tail + (j - head);
    Elem<T>::st(out + i, swish_grad_f32(Elem<T>::ld(grad + i), Elem<T>::ld(x + i), beta));
  }
}

template <typename T>
cudaError_t run(const void* grad_v, const void* x_v, float beta, void* out_v, int64_t n, cudaStream_t stream) {
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
    swish_grad_vec_kernel<T><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(grad + head), reinterpret_cast<const uint4*>(x + head),
        reinterpret_cast<uint4*>(out + head), nvec, beta);
  }
  const int64_t rest = head + (n - tail);
  if (rest > 0) {
    int64_t blocks = (rest + kThreads - 1) / kThreads;
    if (blocks > 4096) blocks = 4096;
    swish_grad_scalar_kernel<T><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(grad, x, out, head, tail,
                                                                                        n, beta);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swish_grad(const void* grad, const void* x, float beta, void* grad_x, int64_t n, int dtype,
                              cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  switch (dtype) {
    case 0: return run<float>(grad, x, beta, grad_x, n, stream);
    case 1: return run<__half>(grad, x, beta, grad_x, n, stream);
    default: return run<__nv_bfloat16>(grad, x, beta, grad_x, n, stream);
  }
}

}  // namespace swg
