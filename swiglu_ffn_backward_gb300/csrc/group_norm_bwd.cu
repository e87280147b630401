// GroupNorm backward: dx, dgamma, dbeta for x, dy of shape [N, C, HxW] (NCHW
// with the spatial dimensions flattened) and gamma of shape [C].
//
// Source: "Beyond automatic differentiation: efficient custom backward
// operators in Ascend C", GroupNorm section: revised version 3.1 (the formula,
// gamma inside the group sums) and 3.2 (groups processed independently, the
// statistics recomputed from x in the backward). With m = (C / G) HxW elements
// per (sample, group), mu and the biased var over the group,
// rstd = 1 / sqrt(var + eps) and x_hat = (x - mu) rstd:
//   dx       = rstd (gamma_c dy - A / m - x_hat B / m),  A = sum gamma dy,  B = sum gamma dy x_hat
//   dgamma_c = sum over samples and positions of dy x_hat,  dbeta_c = the same sum of dy
//
// One cluster of S CTAs (S <= 8) per (sample, group). CTA k of the cluster owns
// a contiguous slice of the group and brings its x and dy into shared memory
// with bulk copies, in up to two parts with one mbarrier each (pass 1 starts on
// the first part while the others arrive), so HBM sees each input once:
//   pass 1    shifted sums, shift K = the group's first x (the shifted-data
//             variance of Chan, Golub and LeVeque, "Algorithms for computing the
//             sample variance: analysis and recommendations", 1983):
//             sum(x - K), sum((x - K)^2), sum(gamma dy), sum(gamma dy (x - K)),
//             and per channel sum(dy), sum(dy (x - K));
//   exchange  the four group sums of every warp of every CTA, added in the same
//             fixed order by every warp (the same value in all of them); the
//             persistent kernel pushes them into each CTA's shared memory with
//             st.async (an mbarrier counts the bytes in), the per-group kernel
//             reads them through distributed shared memory after a cluster
//             barrier; the coefficients are formed in fp32 (this part's FP64
//             rate is a small fraction of its FP32 rate, and this step is on
//             every CTA's critical path);
//   pass 2    dx = (rstd gamma_c) dy + c3 (x - K) + c2', c2' = c2 - c3 d,
//             d = mu - K, written over x in shared memory and stored with bulk
//             copies.
// Both passes work on element pairs with the packed fp32x2 operations. A slice
// longer than the shared-memory stage is taken stage by stage and read again
// for pass 2. Tensors whose groups do not start on 16-byte boundaries take
// plain loads and stores. dgamma, dbeta: the per-(sample, group, slice,
// channel, warp) partials and the per-(sample, group) d and rstd go to the
// workspace; a second kernel adds each sample's partials in fp32 and the
// samples in fp64, in a fixed order, so every output is bitwise reproducible.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
static_assert((kThreads & (kThreads - 1)) == 0, "items are dealt to threads by residue");
constexpr int kParts = 2;                  // bulk-copy parts per stage, one mbarrier each (measured: 2 over 4 and 1)
constexpr int kStageBytes = 96 * 1024;     // largest x and dy stage (slices longer than it are streamed)
constexpr int kSliceBytes = 48 * 1024;     // target x and dy bytes per CTA (measured: 48 KB over 24 and 12)
constexpr int kMinBlocks = 1024 / kThreads;  // resident CTAs per SM the register budget is set for
constexpr int kMaxCluster = 8;             // portable cluster size
constexpr int64_t kMinSlice = 2048;        // elements: smaller slices do not pay for the cluster exchange
constexpr int kPipeSliceBytes = 56 * 1024;     // persistent form: target x and dy bytes per buffer
constexpr int kPipeMaxSliceBytes = 56 * 1024;  // persistent form: largest buffer (two per CTA)

enum : int { kPlain = 0, kBulk = 1, kBulkVec = 2 };

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// two adjacent 16-bit elements (one 32-bit word) <-> a float2; for fp32 a pair of words
__device__ __forceinline__ float2 pair_f(uint32_t u, __half) {
  __half2 h;
  memcpy(&h, &u, 4);
  return __half22float2(h);
}
__device__ __forceinline__ float2 pair_f(uint32_t u, __nv_bfloat16) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ uint32_t pair_t(float2 v, __half) {
  const __half2 h = __floats2half2_rn(v.x, v.y);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}
__device__ __forceinline__ uint32_t pair_t(float2 v, __nv_bfloat16) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Thread t takes the items i = t (mod kThreads) of a slice in every channel segment, so the items of
// a slice spread evenly over the warps whatever the segments' lengths: the first such item at or after s.
__device__ __forceinline__ int first_of_class(int s) {
  return s + ((static_cast<int>(threadIdx.x) - s) & (kThreads - 1));
}

// The 16-byte vectors of one word quadruple: the pass-1 and pass-2 loops work on element pairs with
// the packed fp32x2 operations (__fadd2_rn, __ffma2_rn: one instruction for two lanes of fp32), so the
// sums below hold the even and the odd elements of each pair in .x and .y.
//
// pass-1 sums over stage-local [s, e) of one channel (vectorised: s, e multiples of the vector)
template <typename T, bool kVec>
__device__ __forceinline__ void acc_range(const T* xs, const T* ds, int s, int e, float K, float2& sx, float2& sxx,
                                          float2& sd, float2& se) {
  if (kVec) {
    constexpr int V = 16 / static_cast<int>(sizeof(T));
    const float2 nK = make_float2(-K, -K);
    for (int v = first_of_class(s / V); v < e / V; v += kThreads) {
      const uint4 ux = reinterpret_cast<const uint4*>(xs)[v];
      const uint4 ud = reinterpret_cast<const uint4*>(ds)[v];
      const uint32_t wx[4] = {ux.x, ux.y, ux.z, ux.w}, wd[4] = {ud.x, ud.y, ud.z, ud.w};
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 xk = __fadd2_rn(pair_f(wx[i], T()), nK), dv = pair_f(wd[i], T());
          sx = __fadd2_rn(sx, xk);
          sxx = __ffma2_rn(xk, xk, sxx);
          sd = __fadd2_rn(sd, dv);
          se = __ffma2_rn(dv, xk, se);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 xk = __fadd2_rn(make_float2(__uint_as_float(wx[2 * i]), __uint_as_float(wx[2 * i + 1])), nK);
          const float2 dv = make_float2(__uint_as_float(wd[2 * i]), __uint_as_float(wd[2 * i + 1]));
          sx = __fadd2_rn(sx, xk);
          sxx = __ffma2_rn(xk, xk, sxx);
          sd = __fadd2_rn(sd, dv);
          se = __ffma2_rn(dv, xk, se);
        }
      }
    }
  } else {
    for (int i = first_of_class(s); i < e; i += kThreads) {
      const float xk = to_f(xs[i]) - K, dv = to_f(ds[i]);
      sx.x += xk;
      sxx.x = fmaf(xk, xk, sxx.x);
      sd.x += dv;
      se.x = fmaf(dv, xk, se.x);
    }
  }
}

// pass 2 over stage-local [s, e) of one channel: dx = aj dy + c3 (x - K) + c2', c2' = c2 - c3 d, written
// over x
template <typename T, bool kVec>
__device__ __forceinline__ void dx_range(T* xs, const T* ds, int s, int e, float K, float aj, float d, float c2,
                                         float c3) {
  const float c2d = fmaf(-c3, d, c2);
  if (kVec) {
    constexpr int V = 16 / static_cast<int>(sizeof(T));
    const float2 nK = make_float2(-K, -K), a2 = make_float2(aj, aj), c3v = make_float2(c3, c3),
                 c2v = make_float2(c2d, c2d);
    for (int v = first_of_class(s / V); v < e / V; v += kThreads) {
      const uint4 ux = reinterpret_cast<const uint4*>(xs)[v];
      const uint4 ud = reinterpret_cast<const uint4*>(ds)[v];
      const uint32_t wx[4] = {ux.x, ux.y, ux.z, ux.w}, wd[4] = {ud.x, ud.y, ud.z, ud.w};
      uint32_t wo[4];
      if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 xk = __fadd2_rn(pair_f(wx[i], T()), nK);
          wo[i] = pair_t(__ffma2_rn(a2, pair_f(wd[i], T()), __ffma2_rn(c3v, xk, c2v)), T());
        }
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 xk = __fadd2_rn(make_float2(__uint_as_float(wx[2 * i]), __uint_as_float(wx[2 * i + 1])), nK);
          const float2 o = __ffma2_rn(a2, make_float2(__uint_as_float(wd[2 * i]), __uint_as_float(wd[2 * i + 1])),
                                      __ffma2_rn(c3v, xk, c2v));
          wo[2 * i] = __float_as_uint(o.x);
          wo[2 * i + 1] = __float_as_uint(o.y);
        }
      }
      reinterpret_cast<uint4*>(xs)[v] = make_uint4(wo[0], wo[1], wo[2], wo[3]);
    }
  } else {
    for (int i = first_of_class(s); i < e; i += kThreads)
      xs[i] = from_f<T>(fmaf(aj, to_f(ds[i]), fmaf(c3, to_f(xs[i]) - K, c2d)));
  }
}

struct GnArgs {
  const void* x;
  const void* dy;
  const void* gamma;  // null: gamma = 1
  void* dx;
  float* stats;       // [N G][2]: d = mu - K, rstd        (null when dgamma, dbeta are not wanted)
  float* part;        // [N G][S][Cg][warps][2]: sum dy, sum dy (x - K) per channel and warp (null likewise)
  int64_t hw;         // HxW
  int64_t m;          // Cg HxW
  int64_t slice;      // elements per CTA (multiple of 8)
  int64_t stage;      // shared-memory stage in elements per tensor (multiple of 8)
  int cg;             // channels per group
  int groups;         // G
  int S;              // cluster size
  float eps;
  float inv_m;        // 1 / m, rounded once
  uint32_t* status;
};

// The group's coefficients from the cluster's per-warp sums, computed by every
// warp (the same inputs in the same order give the same values in all warps,
// so no block barrier is needed to share them). After the cluster barrier that
// follows the writes of ws[warp][0..3] = sum(x - K), sum((x - K)^2),
// sum(gamma dy), sum(gamma dy (x - K)) in every CTA of the cluster.
struct GnCoef {
  float d, c1, c2, c3;  // d = mu - K, c1 = rstd; dx = (c1 gamma_c) dy + c2 + c3 ((x - K) - d)
};
// the coefficients from the group sums v0 = sum(x - K), v1 = sum((x - K)^2), v2 = sum(gamma dy),
// v3 = sum(gamma dy (x - K))
__device__ __forceinline__ GnCoef make_coef(float v0, float v1, float v2, float v3, const GnArgs& a) {
  GnCoef c;
  c.d = v0 * a.inv_m;                                         // mu - K
  const float var = fmaxf(fmaf(v1, a.inv_m, -c.d * c.d), 0.0f);  // biased
  c.c1 = rsqrtf(var + a.eps);                                 // rstd
  const float B = c.c1 * fmaf(-c.d, v2, v3);                  // sum gamma dy x_hat
  c.c2 = -c.c1 * v2 * a.inv_m;
  c.c3 = -c.c1 * c.c1 * B * a.inv_m;
  return c;
}
__device__ __forceinline__ GnCoef cluster_coef(const float (*ws)[4], const GnArgs& a) {
  const int lane = threadIdx.x & 31;
  float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
  for (int p = lane; p < a.S * kWarps; p += 32) {  // (rank, warp) pairs, fixed assignment to lanes
    const uint32_t r = static_cast<uint32_t>(p / kWarps);
    const int w = p % kWarps;
    const float t0 = ld_cluster_f32(&ws[w][0], r), t1 = ld_cluster_f32(&ws[w][1], r);
    const float t2 = ld_cluster_f32(&ws[w][2], r), t3 = ld_cluster_f32(&ws[w][3], r);
    v0 += t0;
    v1 += t1;
    v2 += t2;
    v3 += t3;
  }
  return make_coef(warp_sum(v0), warp_sum(v1), warp_sum(v2), warp_sum(v3), a);
}

// channel j closes (ends, or the slice ends inside it): gamma-weight the thread's sums into the
// group sums; the warp's channel partials go to the workspace
__device__ __forceinline__ void close_channel(int j, float gj, float* part, float2& sd2, float2& se2, float& ga,
                                              float& ge) {
  const float sd = sd2.x + sd2.y, se = se2.x + se2.y;
  ga = fmaf(gj, sd, ga);
  ge = fmaf(gj, se, ge);
  if (part != nullptr) {
    const float D = warp_sum(sd), E = warp_sum(se);
    if ((threadIdx.x & 31) == 0) {
      float* q = part + (static_cast<int64_t>(j) * kWarps + (threadIdx.x >> 5)) * 2;
      q[0] = D;
      q[1] = E;
    }
  }
  sd2 = make_float2(0.f, 0.f);
  se2 = make_float2(0.f, 0.f);
}

// One cluster per (sample, group); slices longer than the stage are streamed
// (read again for pass 2); misaligned groups take plain loads and stores.
template <typename T, int kMode>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gn_bwd_kernel(const GnArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  T* xs = reinterpret_cast<T*>(smem);
  T* ds = reinterpret_cast<T*>(smem + a.stage * static_cast<int64_t>(sizeof(T)));
  __shared__ __align__(8) uint64_t bar[kParts];
  __shared__ float wsum[kWarps][4];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t grp = blockIdx.x / a.S;
  const int g = static_cast<int>(grp % a.groups);
  const int64_t base = grp * a.m;
  const T* xg = static_cast<const T*>(a.x) + base;
  const T* dg = static_cast<const T*>(a.dy) + base;
  T* og = static_cast<T*>(a.dx) + base;
  const T* gam = a.gamma != nullptr ? static_cast<const T*>(a.gamma) + static_cast<int64_t>(g) * a.cg : nullptr;
  const int64_t lo = min(a.m, static_cast<int64_t>(rank) * a.slice);
  const int64_t hi = min(a.m, lo + a.slice);
  const int64_t nst = (hi - lo + a.stage - 1) / a.stage;  // stages of this slice
  const float K = to_f(xg[0]);
  float* part = a.part != nullptr ? a.part + (grp * a.S + rank) * static_cast<int64_t>(a.cg) * kWarps * 2 : nullptr;

  if (kMode != kPlain && tid == 0) {
    for (int p = 0; p < kParts; ++p) mbar_init(&bar[p], 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;  // bit p: parity of the next completion of bar[p]
  bool timed_out = false;

  // stage [c0, c0 + clen) of the group -> xs, ds; parts of plen elements (multiple of 8)
  auto plen_of = [&](int64_t clen) -> int64_t {
    if (kMode == kPlain) return clen;
    const int64_t q = (clen + kParts - 1) / kParts;
    return (q + 7) & ~int64_t(7);
  };
  auto issue_stage = [&](int64_t c0, int64_t clen) {
    if (kMode == kPlain) {
      for (int64_t i = tid; i < clen; i += kThreads) {
        xs[i] = xg[c0 + i];
        ds[i] = dg[c0 + i];
      }
      __syncthreads();
    } else if (tid == 0) {
      const int64_t plen = plen_of(clen);
      for (int p = 0; p < kParts; ++p) {
        const int64_t s0 = p * plen, s1 = min(clen, s0 + plen);
        if (s0 >= s1) break;
        const uint32_t bytes = static_cast<uint32_t>((s1 - s0) * static_cast<int64_t>(sizeof(T)));
        mbar_arrive_expect_tx(&bar[p], 2 * bytes);
        bulk_g2s(xs + s0, xg + c0 + s0, bytes, &bar[p]);
        bulk_g2s(ds + s0, dg + c0 + s0, bytes, &bar[p]);
      }
    }
  };
  auto wait_part = [&](int p) {
    if (kMode == kPlain) return;
    if (!mbar_wait(&bar[p], (phase >> p) & 1u)) timed_out = true;
    phase ^= 1u << p;
  };

  // ---------------------------------------------------------------- pass 1
  // Channels are tracked incrementally (no integer division in the loops): j is
  // the channel at stage-local position s, jend the stage-local end of j. The
  // open channel's sums stay in registers across stages.
  float2 sx2 = make_float2(0.f, 0.f), sxx2 = sx2, sd = sx2, se = sx2;
  float ga = 0.f, ge = 0.f;
  bool open = false;
  int j = 0;
  for (int64_t st = 0; st < nst; ++st) {
    const int64_t c0 = lo + st * a.stage;
    const int clen = static_cast<int>(min(a.stage, hi - c0));
    if (st > 0) __syncthreads();  // everyone is done with the previous stage
    issue_stage(c0, clen);
    const int plen = static_cast<int>(plen_of(clen));
    j = static_cast<int>(c0 / a.hw);
    int64_t jend = (j + 1) * a.hw - c0;
    for (int p = 0; p * plen < clen; ++p) {
      wait_part(p);
      const int s1 = min(clen, (p + 1) * plen);
      for (int s = p * plen; s < s1;) {
        const int e = static_cast<int>(min(static_cast<int64_t>(s1), jend));
        acc_range<T, kMode == kBulkVec>(xs, ds, s, e, K, sx2, sxx2, sd, se);
        open = true;
        if (e == jend) {
          close_channel(j, gam != nullptr ? to_f(gam[j]) : 1.0f, part, sd, se, ga, ge);
          open = false;
          ++j;
          jend += a.hw;
        }
        s = e;
      }
    }
  }
  if (open) close_channel(j, gam != nullptr ? to_f(gam[j]) : 1.0f, part, sd, se, ga, ge);  // the slice ends in j

  // ---------------------------------------------------------------- exchange
  const float sx = warp_sum(sx2.x + sx2.y);
  const float sxx = warp_sum(sxx2.x + sxx2.y);
  ga = warp_sum(ga);
  ge = warp_sum(ge);
  if (lane == 0) {
    wsum[warp][0] = sx;
    wsum[warp][1] = sxx;
    wsum[warp][2] = ga;
    wsum[warp][3] = ge;
  }
  cluster_sync();  // every warp's sums in every CTA are written
  const GnCoef cf = cluster_coef(wsum, a);
  if (a.stats != nullptr && rank == 0 && tid == 0) {
    a.stats[2 * grp] = cf.d;
    a.stats[2 * grp + 1] = cf.c1;
  }

  // ---------------------------------------------------------------- pass 2
  for (int64_t st = 0; st < nst; ++st) {
    const int64_t c0 = lo + st * a.stage;
    const int clen = static_cast<int>(min(a.stage, hi - c0));
    const bool reload = nst > 1;
    if (reload) {
      if (kMode != kPlain && tid == 0) bulk_wait_read<0>();  // the previous stage's stores have read xs
      __syncthreads();
      issue_stage(c0, clen);
    }
    const int plen = static_cast<int>(plen_of(clen));
    int jj = static_cast<int>(c0 / a.hw);
    int64_t jend = (jj + 1) * a.hw - c0;
    float aj = cf.c1 * (gam != nullptr ? to_f(gam[jj]) : 1.0f);
    for (int p = 0; p * plen < clen; ++p) {
      if (reload) wait_part(p);
      const int s1 = min(clen, (p + 1) * plen);
      for (int s = p * plen; s < s1;) {
        const int e = static_cast<int>(min(static_cast<int64_t>(s1), jend));
        dx_range<T, kMode == kBulkVec>(xs, ds, s, e, K, aj, cf.d, cf.c2, cf.c3);
        if (e == jend) {
          ++jj;
          jend += a.hw;
          if (jj < a.cg) aj = cf.c1 * (gam != nullptr ? to_f(gam[jj]) : 1.0f);
        }
        s = e;
      }
    }
    if (kMode != kPlain) {
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        bulk_s2g(og + c0, xs, static_cast<uint32_t>(clen * static_cast<int>(sizeof(T))));
        bulk_commit();
      }
    } else {
      __syncthreads();
      for (int i = tid; i < clen; i += kThreads) og[c0 + i] = xs[i];
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still read its sums
  if (kMode != kPlain && tid == 0) bulk_wait_read<0>();  // the stores have read shared memory
  if (timed_out && a.status != nullptr) atomicOr(a.status, kStatusTimeout);
}

// bounded wait on a local mbarrier whose phase completes on st.async writes of the cluster's CTAs:
// acquire at cluster scope, so that those writes are visible after it
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  const uint32_t ad = smem_u32(bar);
  auto try_once = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(ad), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (try_once()) return true;
  const long long t0 = clock64();
  while (!try_once()) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}
// the shared-memory address of `p` (a local object) in cluster CTA `rank`
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// st.async into cluster CTA `rank` at the offset of `dst`, completing its bytes on that CTA's mbarrier
// at the offset of `bar`
__device__ __forceinline__ void st_async_f4(const void* dst, const uint64_t* bar, uint32_t rank, float v0, float v1,
                                            float v2, float v3) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr(dst, rank)),
               "f"(v0), "f"(v1), "f"(v2), "f"(v3), "r"(cluster_addr(bar, rank))
               : "memory");
}
// The group's coefficients from the per-warp sums every CTA of the cluster pushed into this CTA's
// slot (xs[rank][warp] = sum(x - K), sum((x - K)^2), sum(gamma dy), sum(gamma dy (x - K))); the same
// lanes take the same (rank, warp) pairs in the same order in every warp and CTA.
__device__ __forceinline__ GnCoef slot_coef(const float4 (*xs)[kWarps], const GnArgs& a) {
  const int lane = threadIdx.x & 31;
  float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
  for (int p = lane; p < a.S * kWarps; p += 32) {
    const float4 t = xs[p / kWarps][p % kWarps];
    v0 += t.x;
    v1 += t.y;
    v2 += t.z;
    v3 += t.w;
  }
  return make_coef(warp_sum(v0), warp_sum(v1), warp_sum(v2), warp_sum(v3), a);
}

// Persistent, double-buffered form for groups whose slices fit two shared-memory buffers (16-byte
// aligned groups): cluster c takes groups c, c + #clusters, ... (its iterations it = 0, 1, ...), group
// it in buffer it & 1. While a group is worked on, the bulk copies of the next group fill the other
// buffer: its dy half at once, its x half once the store of the previous group has read it (the
// store reads only the x half). The next group's shift K and gammas are loaded during this group and
// converted after it, so their latency is off the chain. Exchange: every warp pushes its four group
// sums into slot it & 1 of every CTA of the cluster with st.async; the slot's mbarrier completes when
// all S x 8 have landed, and each warp forms the coefficients from its own shared memory. A slot is
// written again (for group it + 2) only after every CTA has pushed group it + 1, which each of its
// warps does after reading slot it & 1 for group it: two slots suffice.
template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads, 1) gn_bwd_pipe_kernel(const GnArgs a, int64_t items) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t bar[2][kParts];  // copies of buffer b landed
  __shared__ __align__(8) uint64_t xbar[2];         // exchange slot s complete
  __shared__ __align__(16) float4 xsum[2][kMaxCluster][kWarps];

  // the dgamma/dbeta kernel after this one may be scheduled now: it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t ncl = gridDim.x / a.S;
  const int64_t lo = min(a.m, static_cast<int64_t>(rank) * a.slice);
  const int len = static_cast<int>(min(a.m, lo + a.slice) - lo);  // the same slice of every group
  const int plen = len > 0 ? static_cast<int>((((len + kParts - 1) / kParts) + 7) & ~7) : 1;
  const int np = len > 0 ? (len + plen - 1) / plen : 0;
  const int j0 = len > 0 ? static_cast<int>(lo / a.hw) : 0;            // first channel of the slice
  const int64_t jend0 = (static_cast<int64_t>(j0) + 1) * a.hw - lo;     // slice-local end of channel j0
  const int nch = len > 0 ? static_cast<int>((lo + len - 1) / a.hw) - j0 + 1 : 0;  // channels in the slice
  const bool gl_ok = nch <= 32;  // their gammas are held one per lane
  const uint32_t xbytes = static_cast<uint32_t>(a.S * kWarps * sizeof(float4));
  // buffer b: x at smem + 2 b slice, dy at smem + (2 b + 1) slice (elements of T)
  auto xbuf = [&](int b) { return reinterpret_cast<T*>(smem) + 2 * b * a.slice; };
  auto dbuf = [&](int b) { return reinterpret_cast<T*>(smem) + (2 * b + 1) * a.slice; };
  const T* X = static_cast<const T*>(a.x);
  const T* DY = static_cast<const T*>(a.dy);
  const T* GAM = static_cast<const T*>(a.gamma);
  T* DX = static_cast<T*>(a.dx);

  if (tid == 0) {
    for (int b = 0; b < 2; ++b)
      for (int p = 0; p < kParts; ++p) mbar_init(&bar[b][p], 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&xbar[0], xbytes);  // the first two groups
    mbar_arrive_expect_tx(&xbar[1], xbytes);
  }
  cluster_sync();  // every CTA's barriers are set before a peer writes to them
  uint32_t phase = 0;  // bit b * kParts + p: parity of the next completion of bar[b][p]
  bool timed_out = false;

  // thread 0: this CTA's slice of group `item` -> buffer b, dy half (with the barriers' expected bytes
  // for both halves) and x half
  auto issue_dy = [&](int64_t item, int b) {
    const int64_t off = item * a.m + lo;
    for (int p = 0; p < np; ++p) {
      const int s0 = p * plen, s1 = min(len, s0 + plen);
      const uint32_t bytes = static_cast<uint32_t>((s1 - s0) * static_cast<int>(sizeof(T)));
      mbar_arrive_expect_tx(&bar[b][p], 2 * bytes);
      bulk_g2s(dbuf(b) + s0, DY + off + s0, bytes, &bar[b][p]);
    }
  };
  auto issue_x = [&](int64_t item, int b) {
    const int64_t off = item * a.m + lo;
    for (int p = 0; p < np; ++p) {
      const int s0 = p * plen, s1 = min(len, s0 + plen);
      bulk_g2s(xbuf(b) + s0, X + off + s0, static_cast<uint32_t>((s1 - s0) * static_cast<int>(sizeof(T))),
               &bar[b][p]);
    }
  };
  auto gamma_raw = [&](int64_t item) -> T {  // lane i: gamma of channel j0 + i of group `item`
    return (GAM != nullptr && gl_ok && lane < nch) ? GAM[(item % a.groups) * a.cg + j0 + lane] : from_f<T>(1.0f);
  };

  int64_t w = blockIdx.x / a.S;  // this iteration's group
  float K = w < items ? to_f(X[w * a.m]) : 0.0f;
  float gl = w < items ? to_f(gamma_raw(w)) : 1.0f;
  if (tid == 0 && w < items) {
    issue_dy(w, 0);
    issue_x(w, 0);
  }
  for (int it = 0; w < items; w += ncl, ++it) {
    const int b = it & 1;
    const int64_t wn = w + ncl;
    // the next group: its shift and gammas now (converted after this group), its copies
    T k_raw = from_f<T>(0.0f), g_raw = from_f<T>(1.0f);
    if (wn < items) {
      k_raw = X[wn * a.m];
      g_raw = gamma_raw(wn);
      if (tid == 0) {
        issue_dy(wn, b ^ 1);  // the previous group's store reads only the x half of buffer b ^ 1
        bulk_wait_read<0>();
        issue_x(wn, b ^ 1);
      }
    }
    T* xs = xbuf(b);
    const T* ds = dbuf(b);
    const int g = static_cast<int>(w % a.groups);
    const T* gam = GAM != nullptr ? GAM + static_cast<int64_t>(g) * a.cg : nullptr;
    auto gamma_at = [&](int j) -> float {  // the same value in every lane
      const float v = __shfl_sync(0xffffffffu, gl, (j - j0) & 31);
      return gam == nullptr ? 1.0f : gl_ok ? v : to_f(gam[j]);
    };
    float* part = a.part != nullptr ? a.part + (w * a.S + rank) * static_cast<int64_t>(a.cg) * kWarps * 2 : nullptr;

    // pass 1 (no block barrier: channel partials are per warp)
    float2 sx2 = make_float2(0.f, 0.f), sxx2 = sx2, sd = sx2, se = sx2;
    float ga = 0.f, ge = 0.f;
    {
      int j = j0;
      int64_t jend = jend0;
      bool open = false;
      for (int p = 0; p < np; ++p) {
        if (!mbar_wait(&bar[b][p], (phase >> (b * kParts + p)) & 1u)) timed_out = true;
        phase ^= 1u << (b * kParts + p);
        const int s1 = min(len, (p + 1) * plen);
        for (int s = p * plen; s < s1;) {
          const int e = static_cast<int>(min(static_cast<int64_t>(s1), jend));
          acc_range<T, kVec>(xs, ds, s, e, K, sx2, sxx2, sd, se);
          open = true;
          if (e == jend) {
            close_channel(j, gamma_at(j), part, sd, se, ga, ge);
            open = false;
            ++j;
            jend += a.hw;
          }
          s = e;
        }
      }
      if (open) close_channel(j, gamma_at(j), part, sd, se, ga, ge);
    }

    // exchange
    const float sx = warp_sum(sx2.x + sx2.y), sxx = warp_sum(sxx2.x + sxx2.y);
    ga = warp_sum(ga);
    ge = warp_sum(ge);
    if (lane < a.S) st_async_f4(&xsum[b][rank][warp], &xbar[b], static_cast<uint32_t>(lane), sx, sxx, ga, ge);
    if (!mbar_wait_cluster(&xbar[b], static_cast<uint32_t>((it >> 1) & 1))) timed_out = true;
    if (tid == 0 && wn + ncl < items) mbar_arrive_expect_tx(&xbar[b], xbytes);  // slot b again, for group it + 2
    const GnCoef cf = slot_coef(xsum[b], a);
    if (a.stats != nullptr && rank == 0 && tid == 0) {
      a.stats[2 * w] = cf.d;
      a.stats[2 * w + 1] = cf.c1;
    }

    // pass 2: dx over x in buffer b, one bulk store for the slice
    {
      int j = j0;
      int64_t jend = jend0;
      float aj = cf.c1 * (len > 0 ? gamma_at(j) : 1.0f);
      for (int s = 0; s < len;) {
        const int e = static_cast<int>(min(static_cast<int64_t>(len), jend));
        dx_range<T, kVec>(xs, ds, s, e, K, aj, cf.d, cf.c2, cf.c3);
        if (e == jend) {
          ++j;
          jend += a.hw;
          if (j < a.cg) aj = cf.c1 * gamma_at(j);
        }
        s = e;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0 && len > 0) {
        bulk_s2g(DX + w * a.m + lo, xs, static_cast<uint32_t>(len * static_cast<int>(sizeof(T))));
        bulk_commit();
      }
    }
    K = to_f(k_raw);
    gl = to_f(g_raw);
  }
  cluster_sync();  // no CTA leaves while a peer may still read from or write to it
  if (tid == 0) bulk_wait_read<0>();
  if (timed_out && a.status != nullptr) atomicOr(a.status, kStatusTimeout);
}

// dgamma_c = sum_n rstd_n (E_n - d_n D_n),  dbeta_c = sum_n D_n, with D_n, E_n the sums of channel c's
// partials of sample n over the slices k that hold the channel and the warps w (in fp32, k then w in
// order); the samples are added in fp64 (lane i takes n = i, i + 32, ..., then the warp adds its lanes
// in a fixed tree): one warp per channel, bitwise reproducible. Launched as a programmatic dependent
// of the GroupNorm kernel: griddepcontrol.wait returns once that kernel has completed and its writes
// are visible (without the launch attribute it returns at once).
constexpr int kParamThreads = 128;
template <typename T>
__global__ void __launch_bounds__(kParamThreads) gn_param_kernel(const float* __restrict__ stats,
                                                                 const float* __restrict__ part, T* dgamma, T* dbeta,
                                                                 int64_t N, int C, int G, int cg, int S, int64_t hw,
                                                                 int64_t slice) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int c = static_cast<int>((blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (c >= C) return;
  const int g = c / cg, j = c % cg;
  const int64_t k0 = (j * hw) / slice;
  const int64_t k1 = min(static_cast<int64_t>(S - 1), ((j + 1) * hw - 1) / slice);
  double sb = 0.0, sg = 0.0;
  for (int64_t n = lane; n < N; n += 32) {
    const int64_t grp = n * G + g;
    float D = 0.f, E = 0.f;
    for (int64_t k = k0; k <= k1; ++k) {
      // the channel's kWarps (sum dy, sum dy (x - K)) pairs of slice k: 16-byte aligned, two per float4
      const float4* q = reinterpret_cast<const float4*>(part + ((grp * S + k) * cg + j) * kWarps * 2);
#pragma unroll
      for (int i = 0; i < kWarps / 2; ++i) {
        const float4 v = q[i];
        D += v.x;
        E += v.y;
        D += v.z;
        E += v.w;
      }
    }
    const float2 st = *reinterpret_cast<const float2*>(stats + 2 * grp);  // d, rstd
    sb += static_cast<double>(D);
    sg += static_cast<double>(st.y) * (static_cast<double>(E) - static_cast<double>(st.x) * static_cast<double>(D));
  }
  sb = warp_sum(sb);
  sg = warp_sum(sg);
  if (lane == 0) {
    if (dbeta != nullptr) dbeta[c] = from_f<T>(static_cast<float>(sb));
    if (dgamma != nullptr) dgamma[c] = from_f<T>(static_cast<float>(sg));
  }
}

inline size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

template <typename T, int kMode>
cudaError_t launch_mode(const GnArgs& a, int64_t groups_total, cudaStream_t stream) {
  const size_t smem = 2 * static_cast<size_t>(a.stage) * sizeof(T);
  static std::mutex mu;
  static bool attr_set = false;  // the attribute allows the largest stage; set once per instantiation
  std::lock_guard<std::mutex> lk(mu);
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(gn_bwd_kernel<T, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kStageBytes);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups_total * a.S));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gn_bwd_kernel<T, kMode>, a);
}

// clusters of the persistent form that fit on the device at once (cached per instantiation, S and buffer size)
template <typename T, bool kVec>
cudaError_t launch_pipe(const GnArgs& a, int64_t items, cudaStream_t stream) {
  const size_t smem = 4 * static_cast<size_t>(a.slice) * sizeof(T);
  static std::mutex mu;  // guards the attribute flag and the occupancy cache
  static bool attr_set = false;
  static int cached_S = 0, cached_clusters = 0;
  static size_t cached_smem = 0;
  static int cached_dev = -1;
  std::lock_guard<std::mutex> lk(mu);
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(gn_bwd_pipe_kernel<T, kVec>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kPipeMaxSliceBytes);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (cached_S != a.S || cached_smem != smem || cached_dev != dev) {
    cfg.gridDim = dim3(static_cast<unsigned>(a.S));
    int n = 0;
    cudaError_t err = cudaOccupancyMaxActiveClusters(&n, gn_bwd_pipe_kernel<T, kVec>, &cfg);
    if (err != cudaSuccess) return err;
    cached_S = a.S;
    cached_smem = smem;
    cached_dev = dev;
    cached_clusters = n > 0 ? n : 1;
  }
  const int64_t clusters = items < cached_clusters ? items : cached_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * a.S));
  return cudaLaunchKernelEx(&cfg, gn_bwd_pipe_kernel<T, kVec>, a, items);
}

template <typename T>
cudaError_t run(const void* dy, const void* x, const void* gamma, void* dx, void* dgamma, void* dbeta, int64_t N,
                int64_t C, int64_t HxW, int64_t G, float eps, void* ws, cudaStream_t stream) {
  const int sms = device_sm_count();
  const int64_t es = sizeof(T);
  const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(dy) |
                         reinterpret_cast<uintptr_t>(dx)) & 15u) == 0 &&
                       ((C / G) * HxW * es) % 16 == 0;
  const GnPlan pipe = gn_pipe_plan(N, C, HxW, G, static_cast<int>(es), sms);
  const bool use_pipe = aligned && pipe.S > 0;
  const GnPlan plan = use_pipe ? pipe : gn_plan(N, C, HxW, G, static_cast<int>(es), sms);
  const bool params = dgamma != nullptr || dbeta != nullptr;
  GnArgs a;
  a.x = x;
  a.dy = dy;
  a.gamma = gamma;
  a.dx = dx;
  a.stats = params ? static_cast<float*>(ws) : nullptr;
  a.part = params ? reinterpret_cast<float*>(static_cast<char*>(ws) + al256(static_cast<size_t>(N * G) * 8))
                  : nullptr;
  a.hw = HxW;
  a.m = (C / G) * HxW;
  a.slice = plan.slice;
  a.stage = plan.stage;
  a.cg = static_cast<int>(C / G);
  a.groups = static_cast<int>(G);
  a.S = plan.S;
  a.eps = eps;
  a.inv_m = 1.0f / static_cast<float>(a.m);
  a.status = status_word_ptr();
  const bool vec = aligned && HxW % (16 / es) == 0;
  cudaError_t err = use_pipe  ? (vec ? launch_pipe<T, true>(a, N * G, stream) : launch_pipe<T, false>(a, N * G, stream))
                    : vec     ? launch_mode<T, kBulkVec>(a, N * G, stream)
                    : aligned ? launch_mode<T, kBulk>(a, N * G, stream)
                              : launch_mode<T, kPlain>(a, N * G, stream);
  if (err != cudaSuccess || !params) return err;
  const int64_t threads = C * 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((threads + kParamThreads - 1) / kParamThreads));
  cfg.blockDim = dim3(kParamThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gn_param_kernel<T>, static_cast<const float*>(a.stats),
                            static_cast<const float*>(a.part), static_cast<T*>(dgamma), static_cast<T*>(dbeta), N,
                            static_cast<int>(C), static_cast<int>(G), a.cg, a.S, HxW, a.slice);
}

}  // namespace

GnPlan gn_plan(int64_t N, int64_t C, int64_t HxW, int64_t G, int elem_bytes, int num_sms) {
  GnPlan p;
  const int64_t m = (C / G) * HxW, ng = N * G;
  p.stage = kStageBytes / (2 * elem_bytes);
  const int64_t target = kSliceBytes / (2 * elem_bytes);
  int64_t S = (m + target - 1) / target;  // slices of about the target size
  S = S < 1 ? 1 : (S > kMaxCluster ? kMaxCluster : S);
  // more CTAs per group while the grid is under two CTAs per SM and slices stay long
  while (S < kMaxCluster && ng * S < 2 * static_cast<int64_t>(num_sms) && m / (S + 1) >= kMinSlice) ++S;
  p.S = static_cast<int>(S);
  p.slice = (((m + S - 1) / S) + 7) & ~int64_t(7);
  if (p.slice < p.stage) p.stage = p.slice;  // shared memory for one resident slice
  return p;
}

GnPlan gn_pipe_plan(int64_t N, int64_t C, int64_t HxW, int64_t G, int elem_bytes, int num_sms) {
  GnPlan p;
  const int64_t m = (C / G) * HxW, ng = N * G;
  const int64_t target = kPipeSliceBytes / (2 * elem_bytes);
  int64_t S = (m + target - 1) / target;
  S = S < 1 ? 1 : (S > kMaxCluster ? kMaxCluster : S);
  while (S < kMaxCluster && ng * S < 2 * static_cast<int64_t>(num_sms) && m / (S + 1) >= kMinSlice) ++S;
  p.slice = (((m + S - 1) / S) + 7) & ~int64_t(7);
  p.stage = p.slice;
  p.S = p.slice <= kPipeMaxSliceBytes / (2 * elem_bytes) ? static_cast<int>(S) : 0;  // 0: does not fit
  return p;
}

size_t gn_workspace_bytes(int64_t N, int64_t C, int64_t G) {
  // stats [N G][2] + partials [N G][S <= 8][C / G][warps][2], fp32
  return al256(static_cast<size_t>(N * G) * 8) + al256(static_cast<size_t>(N * C) * kMaxCluster * kWarps * 8);
}

cudaError_t launch_group_norm_bwd(const void* dy, const void* x, const void* gamma, void* dx, void* dgamma,
                                  void* dbeta, int64_t N, int64_t C, int64_t HxW, int64_t G, float eps, int dtype,
                                  void* ws, cudaStream_t stream) {
  switch (dtype) {
    case 0: return run<float>(dy, x, gamma, dx, dgamma, dbeta, N, C, HxW, G, eps, ws, stream);
    case 1: return run<__half>(dy, x, gamma, dx, dgamma, dbeta, N, C, HxW, G, eps, ws, stream);
    case 2: return run<__nv_bfloat16>(dy, x, gamma, dx, dgamma, dbeta, N, C, HxW, G, eps, ws, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace swg
