// Forward of the SwiGLU FFN gate, the producer of the backward's inputs:
//   g = x W_g + b_g,  fc = x W_fc + b_fc,  y = SiLU(g) * fc = g * sigma(g) * fc
// Source: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Operator background" (the forward the backward kernels differentiate).
// bf16 operands, fp32 accumulation in TMEM; g and fc are formed in fp32 with
// the bias, y from those fp32 values, and each output is rounded once to bf16.
//
// One persistent tcgen05 GEMM on CTA pairs (clusters of two, one pair per two
// SMs), ten warps per CTA:
//   warp 0 lane 0   TMA producer (both CTAs): for every 64-wide block of K,
//                   this CTA's x rows [128 m x 64 k] (K-major) and its half of
//                   the B operand [64 k x 128 n] (MN-major, two 64x64 boxes):
//                   W_g in the leader, W_fc in the other CTA; a 6-deep ring
//                   running across the pair's tiles, each stage's copies of
//                   both CTAs counted on the leader's barrier
//   warp 1          TMEM allocation (512 columns in each CTA = two accumulator
//                   buffers, each g [128 x 128] | fc [128 x 128]); lane 0 of
//                   the leader issues tcgen05.mma.cta_group::2 (M=256, N=256,
//                   K=16): one instruction computes both products for the
//                   pair's 256 rows, reading each W tile from one CTA only, so
//                   each SM copies half the W bytes of a single-CTA tile
//   warps 2-9       epilogue (both CTAs, each on its own 128 rows; two warps
//                   per TMEM lane quarter, each on half of the tile's columns):
//                   drain the finished buffer while the tensor cores fill the
//                   other one: bias (read through L1, the same address in every
//                   lane), SiLU, and g, fc, y in turn through the warp's two
//                   64-byte-swizzled 32x32 staging blocks, each written out by
//                   a TMA store (rows beyond M and columns beyond N clipped)
// The pair loops over output tiles [256 rows x 128 columns]; with K = 512 a
// tile holds only eight K blocks, so the double-buffered accumulator is what
// keeps the tensor cores busy across tile boundaries.
//
// Every mbarrier wait is bounded; a timeout sets the module status word,
// stops issuing, drains the pair's TMA copies, frees TMEM and returns.
#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {
namespace {

constexpr int BM = 128;   // rows of a tile in each CTA of the pair
constexpr int BN = 128;   // columns of n per product in a tile
constexpr int BK = 64;    // reduction block
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB: this CTA's x rows
constexpr int B_BYTES = BN * BK * 2;   // 16 KB: this CTA's half of [W_g | W_fc]
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr uint32_t kTmemCols = 512;    // two buffers of [g | fc] in each CTA

struct __align__(1024) FwdSmem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint8_t stage[kEpiWarps][2][2048];  // per epilogue warp: two [32 rows x 32 columns] blocks for TMA stores
  uint64_t full[STAGES];     // leader: both CTAs' copies of the stage have landed
  uint64_t empty[STAGES];    // the pair MMAs reading the stage are done (committed to both CTAs)
  uint64_t tmem_full[2];     // the tile's MMAs into this buffer are done (committed to both CTAs)
  uint64_t tmem_empty[2];    // leader: both CTAs' epilogue warps have read this buffer out
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  volatile uint32_t issued, consumed;
};

struct FwdArgs {
  int M, K, N;
  uint32_t* status;
  const uint16_t* bias[2]; // b_g, b_fc [N] or null
  int tiles, tiles_n, nkb; // pair tiles [256 rows x 128 columns], column tiles, K blocks
  long long wait_limit;    // cycles before a pipeline wait gives up
  int64_t stall_at;        // test injection: the producers stop before this ring entry (-1: never)
};

__device__ __forceinline__ void fwd_timeout(FwdSmem& s, uint32_t* status) {
  if (status != nullptr) atomicOr(status, kStatusTimeout);
  s.abort_flag = 1u;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void stg128(uint16_t* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wg,
               const __grid_constant__ CUtensorMap tm_wfc, const __grid_constant__ CUtensorMap tm_g,
               const __grid_constant__ CUtensorMap tm_fc, const __grid_constant__ CUtensorMap tm_y,
               const FwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem& s = *reinterpret_cast<FwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();  // rank in the pair
  const bool leader = crank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tmem_full[i], 1);
      mbar_init(&s.tmem_empty[i], 2 * kEpiWarps);
    }
    s.abort_flag = 0u;
    s.issued = s.consumed = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_wg);
    tma_prefetch_desc(&tm_wfc);
  }
  if (warp == 1) {
    tmem_alloc_pair(&s.tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrival, commit or copy
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const CUtensorMap* tw = leader ? &tm_wg : &tm_wfc;  // this CTA's half of the B operand
      uint32_t gj = 0;
      bool stopped = false;
      for (int t = cluster; t < args.tiles && !s.abort_flag && !stopped; t += nclusters) {
        const int n0 = (t % args.tiles_n) * BN;
        const int m0 = (t / args.tiles_n) * (2 * BM) + BM * static_cast<int>(crank);
        for (int kb = 0; kb < args.nkb && !s.abort_flag; ++kb, ++gj) {
          if (static_cast<int64_t>(gj) == args.stall_at) {
            stopped = true;
            break;
          }
          const int st = gj % STAGES;
          if (gj >= STAGES && !mbar_wait(&s.empty[st], ((gj / STAGES) - 1) & 1, args.wait_limit)) {
            fwd_timeout(s, args.status);
            break;
          }
          // the leader's barrier counts both CTAs' copies of the stage
          if (leader) mbar_arrive_expect_tx(&s.full[st], 2 * (A_BYTES + B_BYTES));
          const uint32_t full = cluster_addr(&s.full[st], 0);
          const int kr = kb * BK;
          tma_load_2d_pair(s.a[st], &tm_x, full, kr, m0);
          tma_load_2d_pair(s.b[st], tw, full, n0, kr);
          tma_load_2d_pair(s.b[st] + 8192, tw, full, n0 + 64, kr);
          s.issued = gj + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      // M = 256 over the pair, A K-major; B = [W_g (leader) | W_fc (other CTA)] MN-major
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, 2 * BN, 0, 1);
      // a release goes to the barrier at the same offset in both CTAs
      auto commit2 = [](uint64_t* bar) {
        umma_commit_pair(cluster_addr(bar, 0));
        umma_commit_pair(cluster_addr(bar, 1));
      };
      uint32_t gj = 0, it = 0;
      bool ok = true;
      for (int t = cluster; t < args.tiles && ok; t += nclusters, ++it) {
        const uint32_t buf = it & 1;
        if (it >= 2) {
          // the epilogue has read this buffer's previous tile out
          if (!mbar_wait(&s.tmem_empty[buf], ((it >> 1) - 1) & 1, args.wait_limit)) {
            fwd_timeout(s, args.status);
            break;
          }
          tc_fence_after();
        }
        const uint32_t d = tmem + buf * 256;  // in each CTA: g at d, fc at d + 128
        for (int kb = 0; kb < args.nkb; ++kb, ++gj) {
          const int st = gj % STAGES;
          if (!mbar_wait(&s.full[st], (gj / STAGES) & 1, args.wait_limit)) {
            fwd_timeout(s, args.status);
            ok = false;
            break;
          }
          s.consumed = gj + 1;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(s.a[st]);
          const uint32_t b_addr = smem_u32(s.b[st]);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
            // D[:, 0:128] = x W_g, D[:, 128:256] = x W_fc, for the rows of each CTA
            umma_pair(d, smem_desc(a_addr + 32 * k, 16, 1024), smem_desc(b_addr + 2048 * k, 8192, 1024), idesc,
                      acc);
          }
          commit2(&s.empty[st]);
        }
        if (ok) commit2(&s.tmem_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    bool dead = false;
    uint32_t it = 0, nb = 0;  // tiles, staged blocks
    for (int t = cluster; t < args.tiles; t += nclusters, ++it) {
      const uint32_t buf = it & 1;
      const int n0 = (t % args.tiles_n) * BN;
      const int m0 = (t / args.tiles_n) * (2 * BM) + BM * static_cast<int>(crank);
      bool ready = false;
      if (!dead && !s.abort_flag) {
        ready = mbar_wait(&s.tmem_full[buf], (it >> 1) & 1, args.wait_limit);
        if (!ready) {
          fwd_timeout(s, args.status);
          dead = true;
        }
      }
      tc_fence_after();
      // tcgen05.ld is warp-collective: decide for the whole warp
      if (__all_sync(0xffffffffu, ready && !s.abort_flag)) {
        const uint32_t d = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * 256;
        const uint32_t stg = smem_u32(s.stage[warp - 2]);
#pragma unroll 1
        for (int c = 2 * ((warp - 2) >> 2); c < 2 * ((warp - 2) >> 2) + 2; ++c) {
          uint32_t vg[32], vf[32];
          tmem_ld_32x32b_x32(d + c * 32, vg);
          tmem_ld_32x32b_x32(d + BN + c * 32, vf);
          tmem_ld_wait();
          const int col = n0 + c * 32;
          uint4 rg[4], rf[4], ry[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // the biases of these 8 columns, the same address in every lane (zeros beyond N, where the
            // store clips)
            const int cb = col + 8 * j;
            uint4 bgv = make_uint4(0u, 0u, 0u, 0u), bfv = bgv;
            if (cb < args.N) {
              if (args.bias[0] != nullptr) bgv = __ldg(reinterpret_cast<const uint4*>(args.bias[0] + cb));
              if (args.bias[1] != nullptr) bfv = __ldg(reinterpret_cast<const uint4*>(args.bias[1] + cb));
            }
            const uint32_t bgw[4] = {bgv.x, bgv.y, bgv.z, bgv.w};
            const uint32_t bfw[4] = {bfv.x, bfv.y, bfv.z, bfv.w};
            uint32_t og[4], of[4], oy[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i0 = 8 * j + 2 * e;
              const float2 g2 = __fadd2_rn(make_float2(__uint_as_float(vg[i0]), __uint_as_float(vg[i0 + 1])),
                                           bf16x2_to_f2(bgw[e]));
              const float2 f2 = __fadd2_rn(make_float2(__uint_as_float(vf[i0]), __uint_as_float(vf[i0 + 1])),
                                           bf16x2_to_f2(bfw[e]));
              const Sig2 sg = sigmoid_pair2(g2);
              const float2 y2 = __fmul2_rn(__fmul2_rn(g2, sg.s), f2);
              og[e] = pack_bf16x2(g2.x, g2.y);
              of[e] = pack_bf16x2(f2.x, f2.y);
              oy[e] = pack_bf16x2(y2.x, y2.y);
            }
            rg[j] = make_uint4(og[0], og[1], og[2], og[3]);
            rf[j] = make_uint4(of[0], of[1], of[2], of[3]);
            ry[j] = make_uint4(oy[0], oy[1], oy[2], oy[3]);
          }
          // each output in turn through the warp's two staging blocks (this lane's row, 64-byte swizzle:
          // 16-byte chunk j ^ ((row >> 1) & 3)), written out by a TMA store that clips rows beyond M and
          // columns beyond N
#pragma unroll
          for (int o = 0; o < 3; ++o, ++nb) {
            uint8_t* blk = s.stage[warp - 2][nb & 1];
            if (nb >= 2) {
              if (lane == 0) bulk_wait_read<1>();  // the store that used this block has read it
              __syncwarp();
            }
            const uint32_t sb = smem_u32(blk) + lane * 64;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              sts128(sb + ((j ^ ((lane >> 1) & 3)) << 4), o == 0 ? rg[j] : (o == 1 ? rf[j] : ry[j]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (m0 + q * 32 < args.M) tma_store_2d(o == 0 ? &tm_g : (o == 1 ? &tm_fc : &tm_y), blk, col, m0 + q * 32);
              bulk_commit();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // this warp has read its rows of the buffer: tell the leader's MMA issuer
        if (leader)
          mbar_arrive(&s.tmem_empty[buf]);
        else
          mbar_arrive_remote(cluster_addr(&s.tmem_empty[buf], 0));
      }
    }
    if (lane == 0) bulk_wait_all();  // every store has landed before the CTA exits
  }

  __syncthreads();
  cluster_sync();  // both CTAs are done with their roles: no more remote arrivals or commits
  if (leader && threadIdx.x == 0) {
    const uint32_t peer_abort = ld_cluster_u32(&s.abort_flag, 1);
    if (s.abort_flag || peer_abort) {
      // drain: copies of either CTA that complete on the leader's barriers must land before
      // either CTA exits
      const uint32_t peer_issued = ld_cluster_u32(&s.issued, 1);
      const uint32_t issued = s.issued > peer_issued ? s.issued : peer_issued;
      for (uint32_t i = s.consumed; i < issued; ++i)
        if (!mbar_wait(&s.full[i % STAGES], (i / STAGES) & 1, args.wait_limit)) break;
    }
  }
  cluster_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd_gemm(const uint16_t* x, const uint16_t* w_g, const uint16_t* w_fc, const uint16_t* b_g,
                            const uint16_t* b_fc, uint16_t* g, uint16_t* fc, uint16_t* y, int64_t M, int64_t K,
                            int64_t N, cudaStream_t stream) {
  CUtensorMap mx, mwg, mwfc, mg, mfc, my;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  if (!encode_tmap_2d_bf16(&mx, x, K, M, static_cast<uint64_t>(K) * 2, BK, BM) ||
      !encode_tmap_2d_bf16(&mwg, w_g, N, K, rs, 64, BK) || !encode_tmap_2d_bf16(&mwfc, w_fc, N, K, rs, 64, BK) ||
      !encode_tmap_2d_bf16(&mg, g, N, M, rs, 32, 32, 64) || !encode_tmap_2d_bf16(&mfc, fc, N, M, rs, 32, 32, 64) ||
      !encode_tmap_2d_bf16(&my, y, N, M, rs, 32, 32, 64))
    return cudaErrorInvalidValue;
  FwdArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.status = status_word_ptr();
  a.bias[0] = b_g;
  a.bias[1] = b_fc;
  const Injection inj = take_injection(4);
  a.wait_limit = inj.wait_limit;
  a.stall_at = inj.stall_at;
  a.tiles_n = static_cast<int>((N + BN - 1) / BN);
  a.tiles = static_cast<int>(((M + 2 * BM - 1) / (2 * BM)) * a.tiles_n);
  a.nkb = static_cast<int>((K + BK - 1) / BK);
  constexpr size_t smem = sizeof(FwdSmem) + 1024;
  static_assert(smem <= 232448, "forward kernel shared memory");
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // one pair per two SMs, looping over the pair tiles
  int clusters = device_sm_count() / 2;
  if (clusters > a.tiles) clusters = a.tiles;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_kernel, mx, mwg, mwfc, mg, mfc, my, a);
}

}  // namespace swg
