// w stage of the SwiGLU-FFN backward as a tcgen05 (TMEM-accumulator) bf16 GEMM
// fed by TMA (the x stage is in xgemm_tc.cu), and the tensor-map, plan and
// status-word helpers the other kernels share.
//
// Source: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Algorithm overview and formulas" item 3 and the w row of "Kernel
// signatures":
//   w stage: dw_g = x^T dg, dw_fc = x^T dfc -- one launch, the two outputs are
//            two tile sets; the reduction runs over M and is split into S
//            chunks whose fp32 partials a second kernel adds in a fixed order.
// bf16 operands, fp32 accumulation in TMEM, one bf16 rounding per output
// ("Dtype conversion flow": matmul accumulates in fp32).
//
// Persistent: one CTA per SM (6 warps) walks the tiles t, t + #CTAs, ... in an
// order that keeps the tiles in flight on shared operands (w_tile). Warp 0 lane 0
// issues TMA loads into a STAGES-deep ring of shared-memory operand tiles that
// runs across tiles; warp 1 owns the TMEM allocation (two 256-column accumulator
// buffers) and lane 0 issues tcgen05.mma (M=128, N=256, K=16 per instruction) and
// tcgen05.commit; warps 2-5 read a finished 128x256 fp32 accumulator out of TMEM
// (each warp its own 32-lane quarter) and store bf16 (or fp32 partials) while the
// tensor core fills the other buffer.
//
// Operand layouts (shared memory, 128-byte swizzle, written by TMA), MN-major:
// the reduction index m is the strided one. A stage holds 96 rows of m (six K=16
// steps): A tile = x[m0:m0+96, k0:k0+128] as two 96x64 boxes (12 KB apart = LBO,
// the stride between 64-element MN chunks), B tile = dg[m0:m0+96, n0:n0+256] as
// four boxes; 8-row k groups 1024 B apart (SBO), +2048 B per K=16 step. Three
// such stages (216 KB) measured faster than four of 64 rows or three of 80.
// Tails of M, K and N are zero-filled by TMA on load and masked on store.
//
// Every mbarrier wait is bounded; on timeout the kernel ORs a flag into the
// module status word, stops issuing, waits (bounded) for its own TMA copies
// and MMAs still in flight, frees TMEM and returns.
#include <atomic>
#include <mutex>

#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {

__device__ uint32_t g_status = 0;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 96;
constexpr int STAGES = 3;
constexpr int BOX = BK * 128;  // one 64-column box of BK rows (a multiple of 1024 B)
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;  // two accumulator buffers of 256 columns

enum Mode : int { kModeW = 1 };

struct __align__(1024) Smem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];   // the tile's MMAs into this buffer are done
  uint64_t tmem_empty[2];  // the epilogue has read this buffer out
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  volatile uint32_t issued;
  volatile uint32_t consumed;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct GemmArgs {
  int M, K, N;
  uint16_t* dw[2];
  float* ws;
  int splits, kb_per, nkb_total;
  int tiles_kw, tiles_nw;  // dw tile grid per problem
  int tiles;               // splits x 2 x tiles_kw x tiles_nw
  int accumulate;          // dw += this call's sums (one rounding of old + new)
};

__device__ __forceinline__ void flag_timeout(Smem& s) {
  atomicOr(&g_status, kStatusTimeout);
  s.abort_flag = 1u;
}

struct WTile {
  int split, prob, m0, n0, kb_begin, nkb;
};

// Tile t's coordinates. CTAs that run at the same time should share operands: within a (split,
// problem) the dw column tiles go in groups of kGroupN, and inside a group the column index runs
// fastest and the row index next, so the ~150 tiles in flight read about kGroupN dg column blocks
// (each shared by every row tile among them) and a band of x column blocks (each shared by the
// group's columns). With the column index fastest over all of N instead, every wave streamed all of
// dg (at M = 16384, K = 4096, N = 14336: 15.8 GB read from DRAM per launch for 1.1 GB of inputs).
__device__ __forceinline__ WTile w_tile(int t, const GemmArgs& args) {
  constexpr int kGroupN = 8;
  const int per_prob = args.tiles_kw * args.tiles_nw;
  WTile w;
  w.split = t / (2 * per_prob);
  t -= w.split * 2 * per_prob;
  w.prob = t / per_prob;
  t -= w.prob * per_prob;
  const int grp = t / (args.tiles_kw * kGroupN);
  const int gsize = min(kGroupN, args.tiles_nw - grp * kGroupN);
  const int within = t - grp * args.tiles_kw * kGroupN;
  w.m0 = (within / gsize) * BM;                      // dw rows (index k)
  w.n0 = (grp * kGroupN + within % gsize) * BN;      // dw columns (index n)
  w.kb_begin = w.split * args.kb_per;
  w.nkb = min(args.nkb_total, w.kb_begin + args.kb_per) - w.kb_begin;
  return w;
}

// Persistent: one CTA per SM walks tiles t, t + #CTAs, ...; the accumulator is
// double-buffered in TMEM (2 x 256 columns), so a tile's epilogue runs while the
// tensor core accumulates the next one, and the operand ring runs across tiles.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tmem_full[i], 1);
      mbar_init(&s.tmem_empty[i], kEpiThreads);
    }
    s.abort_flag = 0u;
    s.issued = 0u;
    s.consumed = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t gj = 0;  // ring entries issued, over all tiles
      bool stop = false;
      for (int t = blockIdx.x; t < args.tiles && !stop; t += gridDim.x) {
        const WTile w = w_tile(t, args);
        const CUtensorMap* tb = w.prob ? &tmB1 : &tmB0;
        for (int i = 0; i < w.nkb; ++i, ++gj) {
          const int st = gj % STAGES;
          if (gj >= STAGES && !mbar_wait(&s.empty[st], ((gj / STAGES) - 1) & 1)) {
            flag_timeout(s);
            stop = true;
            break;
          }
          if (s.abort_flag) {
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&s.full[st], A_BYTES + B_BYTES);
          const int mr = (w.kb_begin + i) * BK;  // reduction rows of M
          tma_load_2d(s.a[st], &tmA0, &s.full[st], w.m0, mr);
          tma_load_2d(s.a[st] + BOX, &tmA0, &s.full[st], w.m0 + 64, mr);
#pragma unroll
          for (int j = 0; j < 4; ++j) tma_load_2d(s.b[st] + j * BOX, tb, &s.full[st], w.n0 + 64 * j, mr);
          s.issued = gj + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 1, 1);  // both operands MN-major
      uint32_t gj = 0, it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < args.tiles && ok; t += gridDim.x, ++it) {
        const WTile w = w_tile(t, args);
        const uint32_t buf = it & 1;
        if (it >= 2) {
          // the epilogue has read this buffer's previous tile out
          if (!mbar_wait(&s.tmem_empty[buf], ((it >> 1) - 1) & 1)) {
            flag_timeout(s);
            break;
          }
          tc_fence_after();
        }
        const uint32_t d = tmem + buf * BN;
        for (int i = 0; i < w.nkb; ++i, ++gj) {
          const int st = gj % STAGES;
          if (!mbar_wait(&s.full[st], (gj / STAGES) & 1)) {
            flag_timeout(s);
            ok = false;
            break;
          }
          s.consumed = gj + 1;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(s.a[st]);
          const uint32_t b_addr = smem_u32(s.b[st]);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d, smem_desc(a_addr + 2048 * k, BOX, 1024), smem_desc(b_addr + 2048 * k, BOX, 1024),
                      idesc, (i > 0 || k > 0) ? 1u : 0u);
          umma_commit(&s.empty[st]);
        }
        umma_commit(&s.tmem_full[buf]);  // committed even after a timeout: the epilogue stops waiting
      }
      // after a timeout the epilogue may have stopped waiting: see every MMA this thread
      // issued complete before TMEM is freed (the buffer of tile it - 1 was committed last)
      if (s.abort_flag && it > 0) mbar_wait(&s.tmem_full[(it - 1) & 1], ((it - 1) >> 1) & 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    bool dead = false;
    uint32_t it = 0;
    for (int t = blockIdx.x; t < args.tiles; t += gridDim.x, ++it) {
      const WTile w = w_tile(t, args);
      const uint32_t buf = it & 1;
      bool ready = false;
      if (!dead && !s.abort_flag) {
        ready = mbar_wait(&s.tmem_full[buf], (it >> 1) & 1);
        if (!ready) {
          flag_timeout(s);
          dead = true;
        }
      }
      tc_fence_after();
      const int r = q * 32 + lane;  // accumulator row
      // tcgen05.ld is warp-collective: decide for the whole warp
      if (__all_sync(0xffffffffu, ready && !s.abort_flag && w.nkb > 0)) {
        const uint32_t d = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(d + c * 32, v);
          tmem_ld_wait();
          const int row = w.m0 + r;
          const int col = w.n0 + c * 32;
          if (row < args.K) {
            if (args.splits == 1) {
              uint16_t* dwp = w.prob ? args.dw[1] : args.dw[0];
              uint4* dst = reinterpret_cast<uint4*>(dwp + static_cast<int64_t>(row) * args.N + col);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if (col + 8 * j < args.N) {
                  float f[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[8 * j + e]);
                  if (args.accumulate) {
                    const uint4 o = dst[j];
                    dst[j] = make_uint4(add_pack_bf16x2(f[0], f[1], o.x), add_pack_bf16x2(f[2], f[3], o.y),
                                        add_pack_bf16x2(f[4], f[5], o.z), add_pack_bf16x2(f[6], f[7], o.w));
                  } else {
                    dst[j] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                        pack_bf16x2(f[6], f[7]));
                  }
                }
              }
            } else {
              float* dst = args.ws + (static_cast<int64_t>(w.split * 2 + w.prob) * args.K + row) * args.N + col;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                if (col + 4 * j < args.N) {
                  reinterpret_cast<uint4*>(dst)[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.tmem_empty[buf]);  // this thread has read its rows of the buffer
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && s.abort_flag) {
    // drain: TMA copies issued but never consumed must land before the CTA exits
    for (uint32_t i = s.consumed; i < s.issued; ++i) {
      if (!mbar_wait(&s.full[i % STAGES], (i / STAGES) & 1)) break;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// dw[p][k][n] = sum_s ws[s][p][k][n] (fixed order), rounded once to bf16; with
// accumulate, the existing dw value is added to the fp32 sum before that rounding.
__global__ void __launch_bounds__(256) w_split_reduce_kernel(const float4* __restrict__ ws, int splits,
                                                             int64_t per_prob4, uint2* __restrict__ dw_g,
                                                             uint2* __restrict__ dw_fc, int accumulate) {
  const int64_t total4 = 2 * per_prob4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 acc = ws[i];
    for (int sp = 1; sp < splits; ++sp) {
      const float4 v = ws[static_cast<int64_t>(sp) * total4 + i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    uint2* dst = i < per_prob4 ? dw_g + i : dw_fc + (i - per_prob4);
    if (accumulate) {
      const uint2 old = *dst;
      *dst = make_uint2(add_pack_bf16x2(acc.x, acc.y, old.x), add_pack_bf16x2(acc.z, acc.w, old.y));
    } else {
      *dst = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

// ---------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

template <int MODE>
cudaError_t prepare_kernel() {
  return cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemBytes));
}

}  // namespace

static CUtensorMapSwizzle swizzle_mode(int bytes) {
  return bytes == 0    ? CU_TENSOR_MAP_SWIZZLE_NONE
         : bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
         : bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                       : CU_TENSOR_MAP_SWIZZLE_128B;
}

bool encode_tmap_2d_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_mode(swizzle_bytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d_bf16(CUtensorMap* tm, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                         const uint32_t box[3], int swizzle_bytes) {
  EncodeFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides[0], strides[1]};
  const cuuint32_t b[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d, st, b, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_mode(swizzle_bytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

WPlan w_plan(int64_t M, int64_t K, int64_t N, int num_sms) {
  WPlan p;
  const int64_t nkb = (M + BK - 1) / BK;
  const int64_t tiles = 2 * ((K + BM - 1) / BM) * ((N + BN - 1) / BN);
  int64_t splits = num_sms / tiles;
  if (splits < 1) splits = 1;
  // keep at least 8 reduction blocks (768 rows) per split
  const int64_t max_by_len = nkb / 8 > 0 ? nkb / 8 : 1;
  if (splits > max_by_len) splits = max_by_len;
  if (splits > 64) splits = 64;
  p.kb_per = nkb > 0 ? (nkb + splits - 1) / splits : 0;
  p.splits = p.kb_per > 0 ? (nkb + p.kb_per - 1) / p.kb_per : 1;
  p.ws_bytes = p.splits > 1 ? static_cast<size_t>(p.splits) * 2 * K * N * sizeof(float) : 0;
  return p;
}

cudaError_t launch_w_gemm(const uint16_t* x, const uint16_t* dg, const uint16_t* dfc, uint16_t* dw_g,
                          uint16_t* dw_fc, int64_t M, int64_t K, int64_t N, void* ws, const WPlan& plan,
                          cudaStream_t stream, bool accumulate) {
  CUtensorMap a0, b0, b1;
  if (!encode_tmap_2d_bf16(&a0, x, K, M, static_cast<uint64_t>(K) * 2, 64, BK) ||
      !encode_tmap_2d_bf16(&b0, dg, N, M, static_cast<uint64_t>(N) * 2, 64, BK) ||
      !encode_tmap_2d_bf16(&b1, dfc, N, M, static_cast<uint64_t>(N) * 2, 64, BK))
    return cudaErrorInvalidValue;
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.dw[0] = dw_g;
  a.dw[1] = dw_fc;
  a.ws = static_cast<float*>(ws);
  a.splits = static_cast<int>(plan.splits);
  a.kb_per = static_cast<int>(plan.kb_per);
  a.nkb_total = static_cast<int>((M + BK - 1) / BK);
  a.tiles_kw = static_cast<int>((K + BM - 1) / BM);
  a.tiles_nw = static_cast<int>((N + BN - 1) / BN);
  a.accumulate = accumulate ? 1 : 0;
  const int64_t tiles = static_cast<int64_t>(plan.splits) * 2 * a.tiles_kw * a.tiles_nw;
  a.tiles = static_cast<int>(tiles);
  cudaError_t e = prepare_kernel<kModeW>();
  if (e != cudaSuccess) return e;
  int64_t grid = device_sm_count();
  if (grid > tiles) grid = tiles;
  tc_gemm_kernel<kModeW><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(a0, a0, b0, b1, a);
  e = cudaGetLastError();
  if (e != cudaSuccess || plan.splits == 1) return e;
  return launch_w_split_reduce(static_cast<const float*>(ws), plan.splits, K, N, dw_g, dw_fc, stream, accumulate);
}

cudaError_t launch_w_split_reduce(const float* ws, int64_t splits, int64_t K, int64_t N, uint16_t* dw_g,
                                  uint16_t* dw_fc, cudaStream_t stream, bool accumulate) {
  const int64_t per_prob4 = K * N / 4;
  int64_t blocks = (2 * per_prob4 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  w_split_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(ws), static_cast<int>(splits), per_prob4, reinterpret_cast<uint2*>(dw_g),
      reinterpret_cast<uint2*>(dw_fc), accumulate ? 1 : 0);
  return cudaGetLastError();
}

namespace {
std::atomic<int> g_inject_kernel{0};
std::atomic<int64_t> g_inject_stall{-1};
std::atomic<long long> g_inject_limit{kWaitLimitCycles};
}  // namespace

void arm_injection(int kernel, int64_t stall_at, long long wait_limit) {
  g_inject_stall.store(stall_at);
  g_inject_limit.store(wait_limit);
  g_inject_kernel.store(kernel);
}

Injection take_injection(int kernel) {
  int expected = kernel;
  if (kernel != 0 && g_inject_kernel.compare_exchange_strong(expected, 0))
    return Injection{g_inject_stall.load(), g_inject_limit.load()};
  return Injection{-1, kWaitLimitCycles};
}

uint32_t* status_word_ptr() {
  static std::mutex mu;
  static uint32_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

cudaError_t read_and_clear_status(uint32_t* out, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

}  // namespace swg
