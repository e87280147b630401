// b stage of the SwiGLU-FFN backward: dg, dfc and the column sums db_g, db_fc.
//
// Source: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Algorithm overview and formulas" items 1-2 and the b-kernel row of
// "Kernel signatures":
//   dg = dy * fc * sigma(g) * (1 + g * (1 - sigma(g)));  dfc = dy * g * sigma(g)
//   db_g = sum over rows of dg;  db_fc = sum over rows of dfc
// bf16 in/out, fp32 math ("Dtype conversion flow").
//
// HBM-bound: reads 3*M*N*2 bytes, writes 2*M*N*2 bytes (+ 4N for db).
// Layout of one CTA (256 threads) over a [rows_per_chunk x 256] block:
//   warp w covers columns (w & 3)*64 .. +63 and row lane-group (w >> 2);
//   lane l covers the 16-byte vector (l & 7) of those 64 columns and row offset
//   (w >> 2)*4 + (l >> 3) within each group of 8 rows.
// Each thread keeps fp32 running sums of its 8 columns over its rows; a
// warp-shuffle across the 4 row lanes and a shared-memory add across the two
// row warps give the CTA's column sums, written as one fp32 partial row per
// row chunk. A second kernel adds the partial rows in a fixed order (fp64
// accumulator) and rounds once to bf16: no bf16 partial accumulation, and the
// result does not depend on scheduling.
#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {
namespace {

constexpr int kThreads = 256;
constexpr int kCols = 256;  // columns per CTA
constexpr int kRowStep = 8; // rows covered by one pass of the CTA

__device__ __forceinline__ void grad8(const uint4& dy, const uint4& g, const uint4& fc, uint4& dg, uint4& dfc,
                                      float (&ag)[8], float (&af)[8]) {
  const uint32_t dyw[4] = {dy.x, dy.y, dy.z, dy.w};
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
  const uint32_t fw[4] = {fc.x, fc.y, fc.z, fc.w};
  uint32_t og[4], of[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 pg, pf;
    swiglu_grad_pair(bf16x2_to_f2(dyw[i]), bf16x2_to_f2(gw[i]), bf16x2_to_f2(fw[i]), pg, pf);
    ag[2 * i] += pg.x;
    ag[2 * i + 1] += pg.y;
    af[2 * i] += pf.x;
    af[2 * i + 1] += pf.y;
    og[i] = pack_bf16x2(pg.x, pg.y);
    of[i] = pack_bf16x2(pf.x, pf.y);
  }
  dg = make_uint4(og[0], og[1], og[2], og[3]);
  dfc = make_uint4(of[0], of[1], of[2], of[3]);
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// dg/dfc null: only the column sums (used when the caller does not want dg, dfc)
template <bool kStore>
__global__ void __launch_bounds__(kThreads) b_stage_kernel(const uint4* __restrict__ dy, const uint4* __restrict__ g,
                                                           const uint4* __restrict__ fc, uint4* __restrict__ dg,
                                                           uint4* __restrict__ dfc, float* __restrict__ partials,
                                                           int64_t M, int64_t N, int64_t rows_per_chunk) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kCols + (warp & 3) * 64 + (lane & 7) * 8;
  const int rofs = (warp >> 2) * 4 + (lane >> 3);
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_chunk;
  const int64_t r1 = min(M, r0 + rows_per_chunk);
  const int64_t nv = N >> 3;  // 16-byte vectors per row

  float ag[8], af[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ag[i] = af[i] = 0.0f;

  if (col < N) {
    const int64_t cv = col >> 3;
    int64_t row = r0 + rofs;
    // eight rows (stride 8) in flight per thread
    for (; row + 7 * kRowStep < r1; row += 8 * kRowStep) {
      uint4 vdy[8], vg[8], vfc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t off = (row + u * kRowStep) * nv + cv;
        vdy[u] = ld_stream(dy + off);
        vg[u] = ld_stream(g + off);
        vfc[u] = ld_stream(fc + off);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4 odg, odfc;
        grad8(vdy[u], vg[u], vfc[u], odg, odfc, ag, af);
        if (kStore) {
          const int64_t off = (row + u * kRowStep) * nv + cv;
          dg[off] = odg;
          dfc[off] = odfc;
        }
      }
    }
    for (; row < r1; row += kRowStep) {
      const int64_t off = row * nv + cv;
      uint4 odg, odfc;
      grad8(ld_stream(dy + off), ld_stream(g + off), ld_stream(fc + off), odg, odfc, ag, af);
      if (kStore) {
        dg[off] = odg;
        dfc[off] = odfc;
      }
    }
  }

  // sum the 4 row lanes of the warp (lanes l, l^8, l^16, l^24 share columns)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ag[i] += __shfl_xor_sync(0xffffffffu, ag[i], 8);
    ag[i] += __shfl_xor_sync(0xffffffffu, ag[i], 16);
    af[i] += __shfl_xor_sync(0xffffffffu, af[i], 8);
    af[i] += __shfl_xor_sync(0xffffffffu, af[i], 16);
  }
  __shared__ float red[2][2][kCols];  // [row warp group][dg|dfc][column]
  if ((lane >> 3) == 0) {
    const int c = (warp & 3) * 64 + (lane & 7) * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      red[warp >> 2][0][c + i] = ag[i];
      red[warp >> 2][1][c + i] = af[i];
    }
  }
  __syncthreads();
  const int t = threadIdx.x;
  const int64_t gc = static_cast<int64_t>(blockIdx.x) * kCols + t;
  if (gc < N) {
    float* prow = partials + static_cast<int64_t>(blockIdx.y) * 2 * N;
    prow[gc] = red[0][0][t] + red[1][0][t];
    prow[N + gc] = red[0][1][t] + red[1][1][t];
  }
}

// db[j] = sum_c partials[c][j], j over the 2N columns (dg's then dfc's); with
// accumulate, the existing db value joins the fp64 sum before the one rounding.
// Block: 32 columns x 32 chunk lanes; lane ty sums chunks ty, ty+32, ... in
// order, then ty 0..31 are added in order: a fixed summation tree.
__global__ void __launch_bounds__(1024) db_reduce_kernel(const float* __restrict__ partials, int64_t chunks,
                                                         int64_t N, uint16_t* __restrict__ db_g,
                                                         uint16_t* __restrict__ db_fc, int accumulate) {
  __shared__ double acc[32][33];
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * 32 + tx;
  const int64_t two_n = 2 * N;
  double s = 0.0;
  if (j < two_n) {
    for (int64_t c = ty; c < chunks; c += 32) s += static_cast<double>(partials[c * two_n + j]);
  }
  acc[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && j < two_n) {
    double t = 0.0;
    for (int k = 0; k < 32; ++k) t += acc[k][tx];
    uint16_t* dst = j < N ? db_g + j : db_fc + (j - N);
    if (accumulate) t += static_cast<double>(__uint_as_float(static_cast<uint32_t>(*dst) << 16));
    const __nv_bfloat16 b = __double2bfloat16(t);
    *dst = *reinterpret_cast<const uint16_t*>(&b);
  }
}

}  // namespace

BPlan b_plan(int64_t M, int64_t N) {
  // One wave: 4 resident CTAs (64 registers a thread) on each of 152 SMs
  // (measured fastest of 1, 2 and 4 waves at M=220000, N=1024); independent
  // of the device so that the workspace query needs no device.
  const int64_t gx = (N + kCols - 1) / kCols;
  int64_t target = 608 / gx;
  if (target < 1) target = 1;
  int64_t rpc = (M + target - 1) / target;
  rpc = (rpc + 7) / 8 * 8;
  if (rpc < 32) rpc = 32;
  BPlan p;
  p.rows_per_chunk = rpc;
  p.chunks = M > 0 ? (M + rpc - 1) / rpc : 0;
  return p;
}

size_t b_workspace_bytes(int64_t M, int64_t N) {
  const BPlan p = b_plan(M, N);
  return static_cast<size_t>(p.chunks) * 2 * static_cast<size_t>(N) * sizeof(float);
}

cudaError_t launch_db_reduce(const float* partials, int64_t chunks, int64_t N, uint16_t* db_g, uint16_t* db_fc,
                             cudaStream_t stream, bool accumulate) {
  const int64_t blocks = (2 * N + 31) / 32;
  db_reduce_kernel<<<static_cast<unsigned>(blocks), 1024, 0, stream>>>(partials, chunks, N, db_g, db_fc,
                                                                       accumulate ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_b_stage(const uint16_t* dy, const uint16_t* g, const uint16_t* fc, uint16_t* dg, uint16_t* dfc,
                           uint16_t* db_g, uint16_t* db_fc, int64_t M, int64_t N, void* ws, cudaStream_t stream,
                           bool accumulate) {
  const BPlan p = b_plan(M, N);
  float* partials = static_cast<float*>(ws);
  dim3 grid(static_cast<unsigned>((N + kCols - 1) / kCols), static_cast<unsigned>(p.chunks));
  if (dg != nullptr) {
    b_stage_kernel<true><<<grid, kThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(dy), reinterpret_cast<const uint4*>(g), reinterpret_cast<const uint4*>(fc),
        reinterpret_cast<uint4*>(dg), reinterpret_cast<uint4*>(dfc), partials, M, N, p.rows_per_chunk);
  } else {
    b_stage_kernel<false><<<grid, kThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(dy), reinterpret_cast<const uint4*>(g), reinterpret_cast<const uint4*>(fc),
        nullptr, nullptr, partials, M, N, p.rows_per_chunk);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_db_reduce(partials, p.chunks, N, db_g, db_fc, stream, accumulate);
}

}  // namespace swg
