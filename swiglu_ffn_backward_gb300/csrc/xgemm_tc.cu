// x stage of the SwiGLU-FFN backward as a persistent tcgen05 GEMM:
//   dx = dg W_g^T + dfc W_fc^T = [dg | dfc] [W_g | W_fc]^T   (reduction length 2N)
// Source: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Algorithm overview and formulas" item 4 and the x row of "Kernel
// signatures"; bf16 operands, fp32 accumulation in TMEM, one bf16 rounding per
// output ("Dtype conversion flow").
//
// One CTA per SM loops over dx tiles [128 rows x 256 columns] (tile t, t +
// gridDim.x, ...). Tensor memory holds two 256-column accumulators, so the
// epilogue of one tile runs while the tensor core accumulates the next:
//   warp 0 lane 0   TMA producer: a 4-deep ring of K-major tiles, A = dg or dfc
//                   [128 m x 64 n], B = W_g or W_fc [256 k x 64 n] (128-byte
//                   swizzle), running across tiles; the reduction walks (dg, W_g)
//                   then (dfc, W_fc), so no concatenated copy is made
//   warp 1          TMEM allocation (512 columns); lane 0 issues tcgen05.mma
//                   (M=128, N=256, K=16) into the tile's accumulator buffer
//   warps 2-5       epilogue: each drains its 32-lane quarter of the finished
//                   buffer in 32 x 32 blocks: bf16 rounding, a 64-byte-swizzled
//                   staging block, one TMA store per block (rows beyond M and
//                   columns beyond K are clipped by the copy engine)
//
// Every mbarrier wait is bounded; on timeout the kernel ORs a flag into the
// module status word, stops issuing, waits (bounded) for its own TMA copies and
// MMAs, frees TMEM and returns.
#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;   // two 256-column accumulators

struct __align__(1024) XSmem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint8_t stage[kEpiThreads / 32][2][2048];  // per epilogue warp: two 32 x 32 bf16 blocks
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];   // the tile's MMAs into this buffer are done
  uint64_t tmem_empty[2];  // the epilogue has read this buffer out
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  volatile uint32_t issued, consumed;
};

struct XArgs {
  int M, K, N;
  uint32_t* status;
  int tiles, tiles_k, nkb_half;
  long long wait_limit;  // cycles before a pipeline wait gives up
  int stall_at;          // test injection: the producer stops before this ring entry (-1: never)
};

__device__ __forceinline__ void x_timeout(XSmem& s, uint32_t* status) {
  if (status != nullptr) atomicOr(status, kStatusTimeout);
  s.abort_flag = 1u;
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 pack8(const uint32_t* v) {
  return make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                    pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                    pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                    pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
}

__global__ void __launch_bounds__(kThreads, 1)
    x_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                  const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                  const __grid_constant__ CUtensorMap tm_dx, const XArgs args) {
  extern __shared__ uint8_t smem_raw[];
  XSmem& s = *reinterpret_cast<XSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = 2 * args.nkb_half;  // reduction blocks per tile: N/64 of (dg, W_g), then of (dfc, W_fc)

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
    s.issued = s.consumed = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
    tma_prefetch_desc(&tm_dx);
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
      uint32_t gj = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < args.tiles && !stop; t += gridDim.x) {
        const int m0 = (t / args.tiles_k) * BM, n0 = (t % args.tiles_k) * BN;
        for (int kb = 0; kb < nkb; ++kb, ++gj) {
          if (s.abort_flag || static_cast<int>(gj) == args.stall_at) {
            stop = true;
            break;
          }
          const int st = gj % STAGES;
          if (gj >= STAGES && !mbar_wait(&s.empty[st], ((gj / STAGES) - 1) & 1, args.wait_limit)) {
            x_timeout(s, args.status);
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&s.full[st], A_BYTES + B_BYTES);
          const bool second = kb >= args.nkb_half;
          const int r0 = (second ? kb - args.nkb_half : kb) * BK;  // reduction offset within N
          tma_load_2d(s.a[st], second ? &tmA1 : &tmA0, &s.full[st], r0, m0);
          tma_load_2d(s.b[st], second ? &tmB1 : &tmB0, &s.full[st], r0, n0);
          s.issued = gj + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 0);  // both operands K-major
      uint32_t gj = 0, it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < args.tiles && ok; t += gridDim.x, ++it) {
        const uint32_t buf = it & 1;
        if (it >= 2) {
          // the epilogue has read this buffer's previous tile out
          if (!mbar_wait(&s.tmem_empty[buf], ((it >> 1) - 1) & 1, args.wait_limit)) {
            x_timeout(s, args.status);
            break;
          }
          tc_fence_after();
        }
        const uint32_t d = tmem + buf * BN;
        for (int kb = 0; kb < nkb; ++kb, ++gj) {
          const int st = gj % STAGES;
          if (!mbar_wait(&s.full[st], (gj / STAGES) & 1, args.wait_limit)) {
            x_timeout(s, args.status);
            ok = false;
            break;
          }
          s.consumed = gj + 1;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(s.a[st]);
          const uint32_t b_addr = smem_u32(s.b[st]);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d, smem_desc(a_addr + 32 * k, 16, 1024), smem_desc(b_addr + 32 * k, 16, 1024), idesc,
                      (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(&s.empty[st]);
        }
        umma_commit(&s.tmem_full[buf]);  // committed even after a timeout: the epilogue stops waiting
      }
      // after a timeout the epilogue may have stopped waiting: see every MMA this thread
      // issued complete before TMEM is freed (the buffer of tile it - 1 was committed last)
      if (s.abort_flag && it > 0) mbar_wait(&s.tmem_full[(it - 1) & 1], ((it - 1) >> 1) & 1, args.wait_limit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    bool dead = false;
    uint32_t it = 0, nb = 0;  // tiles drained, blocks stored by this warp
    for (int t = blockIdx.x; t < args.tiles; t += gridDim.x, ++it) {
      const uint32_t buf = it & 1;
      const int m0 = (t / args.tiles_k) * BM, n0 = (t % args.tiles_k) * BN;
      bool ready = false;
      if (!dead && !s.abort_flag) {
        ready = mbar_wait(&s.tmem_full[buf], (it >> 1) & 1, args.wait_limit);
        if (!ready) {
          x_timeout(s, args.status);
          dead = true;
        }
      }
      tc_fence_after();
      // tcgen05.ld is warp-collective: decide for the whole warp
      if (__all_sync(0xffffffffu, ready && !s.abort_flag)) {
        const uint32_t d = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c, ++nb) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(d + c * 32, v);
          tmem_ld_wait();
          uint8_t* blk = s.stage[warp - 2][nb & 1];
          if (nb >= 2) {
            if (lane == 0) bulk_wait_read<1>();  // the store that used this block has read it
            __syncwarp();
          }
          // this lane's row of the 32 x 32 block, 64-byte swizzle: 16-byte chunk j ^ ((row >> 1) & 3)
          const uint32_t sb = smem_u32(blk) + lane * 64;
#pragma unroll
          for (int j = 0; j < 4; ++j) sts128(sb + ((j ^ ((lane >> 1) & 3)) << 4), pack8(v + 8 * j));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm_dx, blk, n0 + c * 32, m0 + q * 32);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.tmem_empty[buf]);  // this thread has read its rows of the buffer
    }
    if (lane == 0) bulk_wait_all();  // every store has landed before the CTA exits
  }

  __syncthreads();
  if (threadIdx.x == 0 && s.abort_flag) {
    // drain: copies issued but never consumed must land before the CTA exits
    for (uint32_t i = s.consumed; i < s.issued; ++i)
      if (!mbar_wait(&s.full[i % STAGES], (i / STAGES) & 1, args.wait_limit)) break;
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_x_gemm(const uint16_t* dg, const uint16_t* dfc, const uint16_t* w_g, const uint16_t* w_fc,
                          uint16_t* dx, int64_t M, int64_t K, int64_t N, cudaStream_t stream) {
  CUtensorMap a0, a1, b0, b1, mdx;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  if (!encode_tmap_2d_bf16(&a0, dg, N, M, rs, BK, BM) || !encode_tmap_2d_bf16(&a1, dfc, N, M, rs, BK, BM) ||
      !encode_tmap_2d_bf16(&b0, w_g, N, K, rs, BK, BN) || !encode_tmap_2d_bf16(&b1, w_fc, N, K, rs, BK, BN) ||
      !encode_tmap_2d_bf16(&mdx, dx, K, M, static_cast<uint64_t>(K) * 2, 32, 32, 64))
    return cudaErrorInvalidValue;
  XArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.status = status_word_ptr();
  a.tiles_k = static_cast<int>((K + BN - 1) / BN);
  a.nkb_half = static_cast<int>((N + BK - 1) / BK);
  const int64_t tiles = ((M + BM - 1) / BM) * a.tiles_k;
  a.tiles = static_cast<int>(tiles);
  const Injection inj = take_injection(1);
  a.wait_limit = inj.wait_limit;
  a.stall_at = static_cast<int>(inj.stall_at);
  constexpr size_t smem = sizeof(XSmem) + 1024;
  static_assert(smem <= 232448, "x GEMM shared memory");
  cudaError_t e = cudaFuncSetAttribute(x_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int64_t grid = device_sm_count();
  if (grid > tiles) grid = tiles;
  x_gemm_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(a0, a1, b0, b1, mdx, a);
  return cudaGetLastError();
}

}  // namespace swg
