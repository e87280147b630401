// Fused variant of the SwiGLU-FFN backward: the b-stage math runs inside the
// GEMMs' operand producer, so dg and dfc are formed tile by tile in shared
// memory and never written to (or read back from) HBM.
//
// Sources: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Algorithm overview and formulas" items 1-4 (the math of every stage); the
// recompute-instead-of-store principle stated in the Ascend C backward blog
// post (Swish section: recompute sigma in the backward rather than keep it).
//
// Two kernels, both one CTA per SM with ten warps:
//   warp 0 lane 0   TMA producer of the operand ring (W chunks, or x chunks)
//   warp 1          TMEM allocation (512 columns); lane 0 issues tcgen05.mma
//   warps 2-9       transform: load dy, g, fc straight from global memory into
//                   registers (16-byte coalesced loads, one stage ahead of the
//                   math, with an L2 prefetch of the tile a few stages further
//                   ahead), compute dg, dfc in fp32 and store them as bf16 into
//                   a ring of A-operand slots in the 128-byte-swizzled layout
//                   the tensor cores read; then the epilogue, two warps per
//                   32-lane TMEM quarter, one per 256-column accumulator half.
//   The raw inputs never pass through shared memory: only the operand does.
//
// fused x (FX): D = dx[m0:m0+128, k0:k0+512] in two 256-column accumulators.
//   Stages of 64 reduction columns. A = dg or dfc [128 m x 64 n] (K-major),
//   B = W_g / W_fc chunks [256 k x 64 n] (32 KB ring entries). Each dg element
//   is computed once per 512 columns of dx (once when K <= 512); dg, dfc can
//   also be written to HBM as optional outputs. Persistent: each CTA loops
//   over its tiles, and a tile's epilogue waits until the next tile's first
//   stages are in their A slots, so the tensor core restarts right after it.
// fused w (FW): D = [dw_g^T ; dw_fc^T][n0:n0+64, k0:k0+512]: the A operand
//   stacks 64 columns of dg over the same 64 columns of dfc (MN-major; the two
//   8 KB halves of a slot are the two 64-element MN chunks, LBO = 8 KB), so one
//   accumulator pair holds both outputs for all k. Stages of 64 rows of m;
//   B = x [64 m x 256 k] (MN-major). The CTA owns a fixed band of 64 columns
//   for its whole M range, so it also sums dg, dfc over its rows in registers
//   (db column partials, one row per M split). The reduction over M is split
//   into S chunks with fp32 partials and a fixed-order reduce.
//
// Operand sharing: the copy engine serves a bounded number of 128-byte rows
// per clock per SM, and the operand ring (W in FX, x in FW) is the same for
// several CTAs. CTAs are launched in clusters of CS that share it: CTAs of CS
// consecutive m tiles (FX) or n tiles (FW). Each CTA loads 1/CS of every ring
// entry with a cluster-multicast TMA copy that lands in all CS CTAs; an entry
// is released only when all CS CTAs' MMAs are done with it (the release is a
// multicast tcgen05.commit onto a barrier counting CS arrivals).
//
// Every mbarrier wait is bounded; a timeout sets the module status word,
// stops issuing, drains the CTA's own TMA copies and MMAs, frees TMEM and
// returns.
#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {
namespace {

enum FusedMode : int { kFX = 0, kFW = 1 };

constexpr int kThreads = 320;
constexpr int kXThreads = 256;  // transform / epilogue threads (warps 2-9)
constexpr int kClusterX = 4;    // CTAs sharing each W chunk in the fused x kernel (measured: 3% over 2)
constexpr int kClusterW = 4;    // CTAs sharing each x chunk in the fused w kernel
constexpr uint32_t kTmemCols = 512;

template <int MODE>
struct Cfg;
template <>
struct Cfg<kFX> {
  static constexpr int kRows = 128;        // m rows of a stage's tile (64 columns of n)
  static constexpr int kAStages = 3;       // A-operand slots (dg + dfc, 2 x 16 KB each)
  static constexpr int kEntryBytes = 32768;
  static constexpr int kEntries = 4;
  static constexpr int kPrefetch = 8;      // stages prefetched into L2 ahead of the loads
};
template <>
struct Cfg<kFW> {
  static constexpr int kRows = 64;         // m rows of a stage (64 columns of n)
  static constexpr int kAStages = 4;       // A-operand slots (dg | dfc stacked, 16 KB each)
  static constexpr int kEntryBytes = 32768;
  static constexpr int kEntries = 5;
  static constexpr int kPrefetch = 4;
};

template <int MODE>
struct __align__(1024) FSmem {
  using C = Cfg<MODE>;
  static constexpr int kHalf = C::kRows * 128;  // one 64-column bf16 tile (dg or dfc)
  uint8_t ring[C::kEntries][C::kEntryBytes];
  uint8_t aop[C::kAStages][2 * kHalf];          // [dg | dfc]
  uint64_t a_full[C::kAStages];
  uint64_t a_empty[C::kAStages];
  uint64_t ring_full[C::kEntries];
  uint64_t ring_empty[C::kEntries];
  uint64_t accum;      // one phase per tile: the tile's MMAs are done
  uint64_t tmem_free;  // one phase per tile: the epilogue has read the accumulator
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  volatile uint32_t ring_issued, ring_consumed;
};

struct FusedArgs {
  int M, K, N;
  uint32_t* status;
  int tiles_k;  // 512-column blocks of K
  const uint16_t* dy;
  const uint16_t* g;
  const uint16_t* fc;
  // FX
  uint16_t* dx;
  uint16_t* dg_out;
  uint16_t* dfc_out;
  // FW
  uint16_t* dw_g;
  uint16_t* dw_fc;
  float* ws;       // [splits][2][K][N] dw partials (splits > 1)
  float* db_part;  // [splits][2N]
  int splits, kb_per, nkb_total, tiles_n;
  int x3d;  // x entries come from one 3-D box (else 2-D boxes)
  int cluster_tiles;  // work items of CS CTAs; cluster c takes c, c + nclusters, ...
  int accumulate;     // FW: dw, db += this call's sums (one rounding of old + new)
  int mtiles;         // FX: 128-row tiles of M
  long long wait_limit;  // cycles before a pipeline wait gives up
  int64_t stall_at;      // test injection: the producer stops before this ring entry (-1: never)
};

// One CTA's share of one cluster tile.
struct Tile {
  int m0, n0, k0, kt, split, nst, kb_begin, nh, eps;
};

template <int MODE, int CS>
__device__ __forceinline__ Tile tile_of(int ct, uint32_t crank, const FusedArgs& args) {
  Tile t;
  t.m0 = t.n0 = t.split = t.kb_begin = 0;
  if (MODE == kFX) {
    // cluster tile = CS consecutive m tiles at one 512-column block of K
    t.kt = ct % args.tiles_k;
    t.m0 = ((ct / args.tiles_k) * CS + static_cast<int>(crank)) * 128;
    t.nst = (args.N + 63) / 64;  // stages: 64 columns of n each
  } else {
    // cluster tile = CS consecutive 64-column bands of n, one K block, one M split
    const int bands = args.tiles_n / CS;
    t.n0 = ((ct % bands) * CS + static_cast<int>(crank)) * 64;
    const int rest = ct / bands;
    t.kt = rest % args.tiles_k;
    t.split = rest / args.tiles_k;
    t.kb_begin = t.split * args.kb_per;
    t.nst = min(args.nkb_total, t.kb_begin + args.kb_per) - t.kb_begin;  // stages: 64 rows of m each
  }
  t.k0 = t.kt * 512;
  t.nh = (args.K - t.k0) > 256 ? 2 : 1;             // 256-column accumulator halves in use
  t.eps = (MODE == kFX) ? 2 * t.nh : t.nh;          // ring entries per stage
  return t;
}

template <int MODE>
__device__ __forceinline__ void flag_timeout(FSmem<MODE>& s, uint32_t* status) {
  if (status != nullptr) atomicOr(status, kStatusTimeout);
  s.abort_flag = 1u;
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ldg_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void named_sync_transform() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// dg, dfc for 8 elements; adds them to the column sums
__device__ __forceinline__ void grad8_sum(const uint4& dy, const uint4& g, const uint4& fc, uint4& dg, uint4& dfc,
                                          float (&sg)[8], float (&sf)[8]) {
  const uint32_t dyw[4] = {dy.x, dy.y, dy.z, dy.w};
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
  const uint32_t fw[4] = {fc.x, fc.y, fc.z, fc.w};
  uint32_t og[4], of[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 pg, pf;
    swiglu_grad_pair(bf16x2_to_f2(dyw[i]), bf16x2_to_f2(gw[i]), bf16x2_to_f2(fw[i]), pg, pf);
    const float2 ag = __fadd2_rn(make_float2(sg[2 * i], sg[2 * i + 1]), pg);
    const float2 af = __fadd2_rn(make_float2(sf[2 * i], sf[2 * i + 1]), pf);
    sg[2 * i] = ag.x;
    sg[2 * i + 1] = ag.y;
    sf[2 * i] = af.x;
    sf[2 * i + 1] = af.y;
    og[i] = pack_bf16x2(pg.x, pg.y);
    of[i] = pack_bf16x2(pf.x, pf.y);
  }
  dg = make_uint4(og[0], og[1], og[2], og[3]);
  dfc = make_uint4(of[0], of[1], of[2], of[3]);
}

__device__ __forceinline__ uint4 pack8(const uint32_t* v) {
  return make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                    pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                    pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                    pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
}

template <int MODE, int CS>
__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_g,
                 const __grid_constant__ CUtensorMap tm_fc, const __grid_constant__ CUtensorMap tm_b0,
                 const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_out,
                 const FusedArgs args) {
  using S = FSmem<MODE>;
  using C = Cfg<MODE>;
  constexpr int kAS = C::kAStages;
  constexpr int kRE = C::kEntries;
  constexpr int kRows = C::kRows;
  constexpr int kHalf = S::kHalf;
  constexpr int kRPT = kRows / 32;  // rows per transform thread per stage
  extern __shared__ uint8_t smem_raw[];
  S& s = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t crank = CS > 1 ? cluster_ctarank() : 0u;
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << CS) - 1u);
  const int cluster = blockIdx.x / CS;
  const int nclusters = gridDim.x / CS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAS; ++i) {
      mbar_init(&s.a_full[i], kXThreads);
      mbar_init(&s.a_empty[i], 1);
    }
    for (int i = 0; i < kRE; ++i) {
      mbar_init(&s.ring_full[i], 1);
      mbar_init(&s.ring_empty[i], CS);  // released by all CTAs of the cluster
    }
    mbar_init(&s.accum, 1);
    mbar_init(&s.tmem_free, kXThreads);
    s.abort_flag = 0u;
    s.ring_issued = s.ring_consumed = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_dy);
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_fc);
    tma_prefetch_desc(&tm_b0);
    tma_prefetch_desc(&tm_b1);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (CS > 1) cluster_sync();  // every peer's barriers are initialised before any multicast
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ operand producer
    if (lane == 0) {
      uint32_t gj = 0;  // ring entries issued, over all tiles
      bool stopped = false;  // test injection: nothing more is issued
      for (int ct = cluster; ct < args.cluster_tiles && !s.abort_flag && !stopped; ct += nclusters) {
        const Tile tl = tile_of<MODE, CS>(ct, crank, args);
        const int total = tl.nst * tl.eps;
        for (int j = 0; j < total && !s.abort_flag; ++j, ++gj) {
          if (static_cast<int64_t>(gj) == args.stall_at) {
            stopped = true;
            break;
          }
          const int e = gj % kRE;
          if (gj >= kRE && !mbar_wait(&s.ring_empty[e], ((gj / kRE) - 1) & 1, args.wait_limit)) {
            flag_timeout(s, args.status);
            break;
          }
          const int i = j / tl.eps, q = j % tl.eps;
          mbar_arrive_expect_tx(&s.ring_full[e], C::kEntryBytes);  // all CS slices land here
          if (MODE == kFX) {
            const int p = q / tl.nh, h = q % tl.nh;  // W_g / W_fc, k half
            constexpr int kSliceRows = 256 / CS;
            uint8_t* dst = s.ring[e] + crank * kSliceRows * 128;
            const int kr = tl.k0 + 256 * h + static_cast<int>(crank) * kSliceRows;
            if (CS > 1)
              tma_load_2d_mc(dst, p ? &tm_b1 : &tm_b0, &s.ring_full[e], i * 64, kr, kMask);
            else
              tma_load_2d(dst, p ? &tm_b1 : &tm_b0, &s.ring_full[e], i * 64, kr);
          } else {
            const int mrow = (tl.kb_begin + i) * 64;
            const int kk = tl.k0 + 256 * q;
            constexpr int kSliceChunks = 4 / CS;  // 64x64 blocks of the entry this CTA loads
            const int c_begin = static_cast<int>(crank) * kSliceChunks;
            uint8_t* dst = s.ring[e] + c_begin * 8192;
            if (args.x3d) {
              if (CS > 1)
                tma_load_3d_mc(dst, &tm_b0, &s.ring_full[e], 0, mrow, kk / 64 + c_begin, kMask);
              else
                tma_load_3d(dst, &tm_b0, &s.ring_full[e], 0, mrow, kk / 64 + c_begin);
            } else {
#pragma unroll
              for (int c = 0; c < kSliceChunks; ++c) {
                if (CS > 1)
                  tma_load_2d_mc(dst + c * 8192, &tm_b1, &s.ring_full[e], kk + 64 * (c_begin + c), mrow, kMask);
                else
                  tma_load_2d(dst + c * 8192, &tm_b1, &s.ring_full[e], kk + 64 * (c_begin + c), mrow);
              }
            }
          }
          s.ring_issued = gj + 1;
        }
      }
      if (CS > 1 && !s.abort_flag) {
        // the peers' last releases arrive on this CTA's barriers: see them land
        // before this CTA can leave
        for (uint32_t j = gj > static_cast<uint32_t>(kRE) ? gj - kRE : 0u; j < gj; ++j)
          if (!mbar_wait(&s.ring_empty[j % kRE], (j / kRE) & 1, args.wait_limit)) {
            flag_timeout(s, args.status);
            break;
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 256, MODE == kFW, MODE == kFW);
      uint32_t gi = 0, gj = 0, tt = 0;  // A stages, ring entries, tiles consumed
      bool ok = true;
      for (int ct = cluster; ct < args.cluster_tiles && ok; ct += nclusters, ++tt) {
        const Tile tl = tile_of<MODE, CS>(ct, crank, args);
        if (tt > 0) {
          // the previous tile's epilogue must have read the accumulator out
          if (!mbar_wait(&s.tmem_free, (tt - 1) & 1, args.wait_limit)) {
            flag_timeout(s, args.status);
            break;
          }
          tc_fence_after();
        }
        for (int i = 0; i < tl.nst && ok; ++i, ++gi) {
          const int a = gi % kAS;
          if (!mbar_wait(&s.a_full[a], (gi / kAS) & 1, args.wait_limit)) {
            flag_timeout(s, args.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_slot = smem_u32(s.aop[a]);
          for (int q = 0; q < tl.eps; ++q, ++gj) {
            const int e = gj % kRE;
            if (!mbar_wait(&s.ring_full[e], (gj / kRE) & 1, args.wait_limit)) {
              flag_timeout(s, args.status);
              ok = false;
              break;
            }
            s.ring_consumed = gj + 1;
            tc_fence_after();
            const uint32_t b_addr = smem_u32(s.ring[e]);
            if (MODE == kFX) {
              const int p = q / tl.nh, h = q % tl.nh;
              const uint32_t a_addr = a_slot + p * kHalf;  // dg or dfc
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_bf16(tmem + h * 256, smem_desc(a_addr + 32 * k, 16, 1024),
                          smem_desc(b_addr + 32 * k, 16, 1024), idesc, (i > 0 || p > 0 || k > 0) ? 1u : 0u);
            } else {
              const int h = q;
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_bf16(tmem + h * 256, smem_desc(a_slot + 2048 * k, kHalf, 1024),
                          smem_desc(b_addr + 2048 * k, 8192, 1024), idesc, (i > 0 || k > 0) ? 1u : 0u);
            }
            if (CS > 1)
              umma_commit_mc(&s.ring_empty[e], kMask);  // release the entry in every CTA of the cluster
            else
              umma_commit(&s.ring_empty[e]);
          }
          umma_commit(&s.a_empty[a]);
        }
        umma_commit(&s.accum);  // this tile's accumulator is complete
      }
      // after a timeout the epilogue may have stopped waiting: see every MMA this thread
      // issued complete before the CTA frees TMEM (tt accumulator phases were committed)
      if (s.abort_flag && tt > 0) mbar_wait(&s.accum, (tt - 1) & 1, args.wait_limit);
    }
  } else {
    // ------------------------------------------------------------ transform
    const int t = threadIdx.x - 64;  // 0..255
    const int c = t & 7;             // 16-byte chunk of the 64-column tile (8 columns)
    const int rg = t >> 3;           // row group 0..31; rows rg, rg + 32, ...
    const int64_t N64 = args.N;
    // A thread whose wait runs out stops computing ("dead") but keeps taking
    // part in the arrivals and the named barriers.
    bool dead = false;

    // stores one stage's dg, dfc (8 columns x kRPT rows of this thread) into A slot a
    auto store_stage = [&](int a, int row0, int col, bool want_dg, const uint4 (&bdy)[kRPT],
                           const uint4 (&bg)[kRPT], const uint4 (&bfc)[kRPT], float (&cg)[8], float (&cf)[8]) {
      const uint32_t sdg = smem_u32(s.aop[a]);
      const uint32_t sdf = sdg + kHalf;
#pragma unroll
      for (int q = 0; q < kRPT; ++q) {
        const int row = rg + 32 * q;  // row within the tile
        // 128-byte swizzle: the 16-byte chunk index is XORed with row & 7
        const uint32_t off = row * 128 + ((c ^ (row & 7)) << 4);
        uint4 odg, odfc;
        grad8_sum(bdy[q], bg[q], bfc[q], odg, odfc, cg, cf);
        sts128(sdg + off, odg);
        sts128(sdf + off, odfc);
        if (want_dg) {
          const int r = row0 + row;
          if (r < args.M && col < args.N) {
            const int64_t o = static_cast<int64_t>(r) * N64 + col;
            *reinterpret_cast<uint4*>(args.dg_out + o) = odg;
            *reinterpret_cast<uint4*>(args.dfc_out + o) = odfc;
          }
        }
      }
      fence_proxy_async_smem();  // dg, dfc written by this thread -> visible to the tensor core
    };
    auto load_rows = [&](int row0, int col, bool valid, uint4 (&bdy)[kRPT], uint4 (&bg)[kRPT],
                         uint4 (&bfc)[kRPT]) {
#pragma unroll
      for (int q = 0; q < kRPT; ++q) {
        const int row = row0 + rg + 32 * q;
        if (valid && row < args.M && col < args.N) {  // tails read as zeros
          const int64_t o = static_cast<int64_t>(row) * N64 + col;
          bdy[q] = ldg_stream(args.dy + o);
          bg[q] = ldg_stream(args.g + o);
          bfc[q] = ldg_stream(args.fc + o);
        } else {
          bdy[q] = bg[q] = bfc[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    };
    // waits for A slot a to be released by the MMAs of stage st - kAS
    auto acquire_slot = [&](uint32_t st, int a) {
      if (!dead && st >= kAS && !mbar_wait(&s.a_empty[a], ((st / kAS) - 1) & 1, args.wait_limit)) {
        flag_timeout(s, args.status);
        dead = true;
      }
      if (s.abort_flag) dead = true;
    };
    uint4 xdy[kRPT], xg[kRPT], xfc[kRPT], ydy[kRPT], yg[kRPT], yfc[kRPT];

    if constexpr (MODE == kFX) {
      // The CTA's stages form one stream over its tiles: stage st is stage
      // st % nst of the CTA's tile st / nst, and also the global A-stage index.
      // A tile's epilogue runs after the first kAS - 1 stages of the next tile
      // are in their A slots, so the tensor core restarts as soon as the
      // accumulator is drained; the staging buffer of the epilogue's TMA stores
      // is the A slot of the finished tile's last stage, free once its MMAs are.
      const int nst = (args.N + 63) / 64;
      const int ntiles = cluster < args.cluster_tiles ? (args.cluster_tiles - 1 - cluster) / nclusters + 1 : 0;
      const int total = ntiles * nst;
      const int look = nst < kAS - 1 ? nst : kAS - 1;
      auto tile_at = [&](int tix) { return tile_of<MODE, CS>(cluster + tix * nclusters, crank, args); };
      float ug[8], uf[8];  // column sums, unused here
#pragma unroll
      for (int e = 0; e < 8; ++e) ug[e] = uf[e] = 0.0f;

      auto load = [&](int st, uint4 (&bdy)[kRPT], uint4 (&bg)[kRPT], uint4 (&bfc)[kRPT]) {
        const bool valid = st < total;
        const int m0 = valid ? tile_at(st / nst).m0 : 0;
        load_rows(m0, (valid ? (st % nst) * 64 : 0) + c * 8, valid, bdy, bg, bfc);
      };
      auto prefetch = [&](int st) {
        if (st < total) {
          const int m0 = tile_at(st / nst).m0, p0 = (st % nst) * 64;
          tma_prefetch_l2_2d(&tm_dy, p0, m0);
          tma_prefetch_l2_2d(&tm_g, p0, m0);
          tma_prefetch_l2_2d(&tm_fc, p0, m0);
        }
      };
      auto process = [&](int st, const uint4 (&bdy)[kRPT], const uint4 (&bg)[kRPT], const uint4 (&bfc)[kRPT]) {
        const int a = st % kAS;
        acquire_slot(static_cast<uint32_t>(st), a);
        if (!dead) {
          const Tile tl = tile_at(st / nst);
          store_stage(a, tl.m0, (st % nst) * 64 + c * 8, tl.kt == 0 && args.dg_out != nullptr, bdy, bg, bfc, ug,
                      uf);
        }
        mbar_arrive(&s.a_full[a]);
      };
      // tile tix's accumulator -> bf16 dx through staging buffer stg (an A slot)
      auto epilogue = [&](int tix, int stg) {
        const Tile tl = tile_at(tix);
        bool acc_ok = false;
        if (!dead && !s.abort_flag) {
          acc_ok = mbar_wait(&s.accum, tix & 1, args.wait_limit);
          if (!acc_ok) flag_timeout(s, args.status);
        }
        const int q = warp & 3;         // TMEM lane quarter this warp may read
        const int h = (warp - 2) >> 2;  // accumulator half this warp drains
        tc_fence_after();
        // tcgen05.ld is warp-collective: decide for the whole warp
        if (h < tl.nh && __all_sync(0xffffffffu, !dead && acc_ok && !s.abort_flag)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 256 + cc * 32, v);
            tmem_ld_wait();
            // this warp's 32 x 32 block -> a 64-byte-swizzled staging buffer -> one TMA
            // store (rows beyond M and columns beyond K are clipped by the copy engine)
            uint8_t* buf = s.aop[stg] + (warp - 2) * 4096 + (cc & 1) * 2048;
            if (cc >= 2) {
              if (lane == 0) bulk_wait_read<1>();  // the store that used this buffer has read it
              __syncwarp();
            }
            const uint32_t sb = smem_u32(buf) + lane * 64;
#pragma unroll
            for (int j = 0; j < 4; ++j) sts128(sb + ((j ^ ((lane >> 1) & 3)) << 4), pack8(v + 8 * j));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_out, buf, tl.k0 + h * 256 + cc * 32, tl.m0 + q * 32);
              bulk_commit();
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&s.tmem_free);  // this thread has read its part of the accumulator
        // the staging slot is written again by a later stage: every store has read it
        if (lane == 0) bulk_wait_read<0>();
        named_sync_transform();
      };
      auto after = [&](int st) {
        const int tix = st / nst;
        if (tix >= 1 && st % nst + 1 == look) epilogue(tix - 1, (tix * nst - 1) % kAS);
      };

      if (t == 0)
        for (int p = 0; p <= C::kPrefetch; ++p) prefetch(p);
      load(0, xdy, xg, xfc);
      for (int st = 0; st < total; st += 2) {
        // two stages per iteration, alternating register buffers: the loads of the
        // next stage are in flight while this stage is computed (and while an
        // epilogue runs)
        if (t == 0) prefetch(st + 1 + C::kPrefetch);
        load(st + 1, ydy, yg, yfc);
        process(st, xdy, xg, xfc);
        after(st);
        if (st + 1 >= total) break;
        if (t == 0) prefetch(st + 2 + C::kPrefetch);
        load(st + 2, xdy, xg, xfc);
        process(st + 1, ydy, yg, yfc);
        after(st + 1);
      }
      if (ntiles > 0) epilogue(ntiles - 1, (total - 1) % kAS);
      if (lane == 0) bulk_wait_all();  // every store has landed before the CTA exits
    } else {
      uint32_t gi = 0, tt = 0;  // A stages, tiles produced
      for (int ct = cluster; ct < args.cluster_tiles; ct += nclusters, ++tt) {
        const Tile tl = tile_of<MODE, CS>(ct, crank, args);
        const int n0 = tl.n0, k0 = tl.k0, kb_begin = tl.kb_begin, nst = tl.nst, nh = tl.nh, split = tl.split;
        const bool want_db = tl.kt == 0 && args.db_part != nullptr;
        float cg[8], cf[8];  // column sums over the CTA's whole M range
#pragma unroll
        for (int e = 0; e < 8; ++e) cg[e] = cf[e] = 0.0f;

        auto load = [&](int i, uint4 (&bdy)[kRPT], uint4 (&bg)[kRPT], uint4 (&bfc)[kRPT]) {
          load_rows((kb_begin + i) * 64, n0 + c * 8, i < nst, bdy, bg, bfc);
        };
        auto prefetch = [&](int i) {
          if (i < nst) {
            const int p1 = (kb_begin + i) * 64;
            tma_prefetch_l2_2d(&tm_dy, n0, p1);
            tma_prefetch_l2_2d(&tm_g, n0, p1);
            tma_prefetch_l2_2d(&tm_fc, n0, p1);
          }
        };
        auto process = [&](int i, const uint4 (&bdy)[kRPT], const uint4 (&bg)[kRPT], const uint4 (&bfc)[kRPT]) {
          const uint32_t gs = gi + i;  // global A-stage index
          const int a = gs % kAS;
          acquire_slot(gs, a);
          if (!dead) store_stage(a, (kb_begin + i) * 64, n0 + c * 8, false, bdy, bg, bfc, cg, cf);
          mbar_arrive(&s.a_full[a]);
        };

        if (t == 0)
          for (int i = 0; i <= C::kPrefetch; ++i) prefetch(i);
        load(0, xdy, xg, xfc);
        for (int i = 0; i < nst; i += 2) {
          if (t == 0) prefetch(i + 1 + C::kPrefetch);
          load(i + 1, ydy, yg, yfc);
          process(i, xdy, xg, xfc);
          if (i + 1 >= nst) break;
          if (t == 0) prefetch(i + 2 + C::kPrefetch);
          load(i + 2, xdy, xg, xfc);
          process(i + 1, ydy, yg, yfc);
        }

        gi += nst;
        bool acc_ok = false;
        if (!dead && !s.abort_flag) {
          acc_ok = mbar_wait(&s.accum, tt & 1, args.wait_limit);
          if (!acc_ok) flag_timeout(s, args.status);
        }
        if (want_db) {
          // Column sums over the CTA's rows (rows beyond M were read as zeros).
          // Lanes l, l^8, l^16, l^24 share a chunk; the 8 warps are combined
          // through the first A slot, idle once accum has fired.
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            cg[e] += __shfl_xor_sync(0xffffffffu, cg[e], 8);
            cg[e] += __shfl_xor_sync(0xffffffffu, cg[e], 16);
            cf[e] += __shfl_xor_sync(0xffffffffu, cf[e], 8);
            cf[e] += __shfl_xor_sync(0xffffffffu, cf[e], 16);
          }
          named_sync_transform();
          float* scratch = reinterpret_cast<float*>(s.aop[0]);  // [8 warps][8 chunks][16]
          if (lane < 8) {
            float* pp = scratch + ((warp - 2) * 8 + c) * 16;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              pp[e] = cg[e];
              pp[8 + e] = cf[e];
            }
          }
          named_sync_transform();
          if (t < 128) {
            const int which = t >> 6;  // 0: dg, 1: dfc
            const int col = t & 63;
            const int gc = n0 + col;
            if (!dead && acc_ok && gc < args.N) {
              float v = 0.0f;
#pragma unroll
              for (int w = 0; w < 8; ++w) v += scratch[(w * 8 + (col >> 3)) * 16 + which * 8 + (col & 7)];
              args.db_part[static_cast<int64_t>(split) * 2 * args.N + which * args.N + gc] = v;
            }
          }
          named_sync_transform();  // the scratch is read before a later tile's stage reuses the slot
        }

        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        tc_fence_after();
        const int r = q * 32 + lane;    // accumulator row (TMEM lane)
        const int h = (warp - 2) >> 2;  // accumulator half this warp drains
        // tcgen05.ld is warp-collective: decide for the whole warp
        if (h < nh && __all_sync(0xffffffffu, !dead && acc_ok && !s.abort_flag && nst > 0)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 256 + cc * 32, v);
            tmem_ld_wait();
            const int kcol = k0 + h * 256 + cc * 32;
            const int prob = r >> 6;  // lanes 0-63: dw_g, 64-127: dw_fc
            const int n = n0 + (r & 63);
            if (n < args.N) {
              if (args.splits == 1) {
                uint16_t* dst = (prob ? args.dw_fc : args.dw_g) + n;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const int k = kcol + e;
                  if (k < args.K) {
                    uint16_t* d = dst + static_cast<int64_t>(k) * args.N;
                    float val = __uint_as_float(v[e]);
                    if (args.accumulate) val += __uint_as_float(static_cast<uint32_t>(*d) << 16);
                    const __nv_bfloat16 b = __float2bfloat16_rn(val);
                    *d = *reinterpret_cast<const uint16_t*>(&b);
                  }
                }
              } else {
                float* dst = args.ws + static_cast<int64_t>(split * 2 + prob) * args.K * args.N + n;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const int k = kcol + e;
                  if (k < args.K) dst[static_cast<int64_t>(k) * args.N] = __uint_as_float(v[e]);
                }
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&s.tmem_free);  // this thread has read its part of the accumulator
      }  // tile loop
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && s.abort_flag) {
    // drain: ring copies issued but never waited on must land before the CTA exits
    for (uint32_t i = s.ring_consumed; i < s.ring_issued; ++i)
      if (!mbar_wait(&s.ring_full[i % kRE], (i / kRE) & 1, args.wait_limit)) break;
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (CS > 1) cluster_sync();  // no CTA leaves while a peer may still write into it
}

template <int MODE>
constexpr size_t smem_bytes() {
  return sizeof(FSmem<MODE>) + 1024;
}

template <int MODE, int CS>
cudaError_t launch(unsigned grid, cudaStream_t stream, const CUtensorMap& a, const CUtensorMap& b,
                   const CUtensorMap& c, const CUtensorMap& d, const CUtensorMap& e, const CUtensorMap& out,
                   FusedArgs args, bool persistent) {
  constexpr size_t smem = smem_bytes<MODE>();
  static_assert(smem <= 232448, "fused kernel shared memory");
  cudaError_t err = cudaFuncSetAttribute(fused_kernel<MODE, CS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  args.cluster_tiles = static_cast<int>(grid / CS);
  if (persistent) {
    // one resident wave of clusters, each looping over cluster tiles
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, fused_kernel<MODE, CS>, &cfg) == cudaSuccess &&
        max_clusters > 0 && static_cast<unsigned>(max_clusters) * CS < grid)
      cfg.gridDim = dim3(static_cast<unsigned>(max_clusters) * CS);
  }
  return cudaLaunchKernelEx(&cfg, fused_kernel<MODE, CS>, a, b, c, d, e, out, args);
}

inline size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

FwPlan fw_plan(int64_t M, int64_t K, int64_t N, int num_sms) {
  FwPlan p;
  const int64_t nkb = (M + 63) / 64;
  const int64_t tiles = ((N + 63) / 64) * ((K + 511) / 512);
  int64_t splits = num_sms / tiles;
  if (splits < 1) splits = 1;
  const int64_t max_by_len = nkb / 8 > 0 ? nkb / 8 : 1;  // at least 512 rows per split
  if (splits > max_by_len) splits = max_by_len;
  if (splits > 64) splits = 64;
  p.kb_per = nkb > 0 ? (nkb + splits - 1) / splits : 0;
  p.splits = p.kb_per > 0 ? (nkb + p.kb_per - 1) / p.kb_per : 1;
  const size_t dw_part = p.splits > 1 ? static_cast<size_t>(p.splits) * 2 * K * N * sizeof(float) : 0;
  const size_t db_part = static_cast<size_t>(p.splits) * 2 * N * sizeof(float);
  p.ws_bytes = al256(dw_part) + al256(db_part);
  return p;
}

cudaError_t launch_fused_x(const uint16_t* dy, const uint16_t* g, const uint16_t* fc, const uint16_t* w_g,
                           const uint16_t* w_fc, uint16_t* dx, uint16_t* dg, uint16_t* dfc, int64_t M, int64_t K,
                           int64_t N, cudaStream_t stream) {
  constexpr int CS = kClusterX;
  CUtensorMap mdy, mg, mfc, mw0, mw1, mdx;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  if (!encode_tmap_2d_bf16(&mdx, dx, K, M, static_cast<uint64_t>(K) * 2, 32, 32, 64)) return cudaErrorInvalidValue;
  // the raw tensors are only prefetched into L2 here, one stage's box at a time
  if (!encode_tmap_2d_bf16(&mdy, dy, N, M, rs, 64, 128, 0) || !encode_tmap_2d_bf16(&mg, g, N, M, rs, 64, 128, 0) ||
      !encode_tmap_2d_bf16(&mfc, fc, N, M, rs, 64, 128, 0) ||
      !encode_tmap_2d_bf16(&mw0, w_g, N, K, rs, 64, 256 / CS) ||
      !encode_tmap_2d_bf16(&mw1, w_fc, N, K, rs, 64, 256 / CS))
    return cudaErrorInvalidValue;
  FusedArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.status = status_word_ptr();
  a.tiles_k = static_cast<int>((K + 511) / 512);
  a.dy = dy;
  a.g = g;
  a.fc = fc;
  a.dx = dx;
  a.dg_out = dg;
  a.dfc_out = dfc;
  const Injection inj = take_injection(2);
  a.wait_limit = inj.wait_limit;
  a.stall_at = inj.stall_at;
  const int64_t mclusters = ((M + 127) / 128 + CS - 1) / CS;  // tail CTAs run on zero-filled rows
  return launch<kFX, CS>(static_cast<unsigned>(mclusters * CS * a.tiles_k), stream, mdy, mg, mfc, mw0, mw1, mdx, a,
                         true);
}

namespace {

// the FW kernel alone: fp32 split partials into dw_part / db_part when plan.splits > 1, else bf16 dw
// straight into dw_g, dw_fc (db always as partials)
cudaError_t launch_fw_kernel(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                             uint16_t* dw_g, uint16_t* dw_fc, int64_t M, int64_t K, int64_t N, float* dw_part,
                             float* db_part, const FwPlan& plan, cudaStream_t stream, bool accumulate) {
  CUtensorMap mdy, mg, mfc, mx2, mx3;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  if (!encode_tmap_2d_bf16(&mdy, dy, N, M, rs, 64, 64) || !encode_tmap_2d_bf16(&mg, g, N, M, rs, 64, 64) ||
      !encode_tmap_2d_bf16(&mfc, fc, N, M, rs, 64, 64) ||
      !encode_tmap_2d_bf16(&mx2, x, K, M, static_cast<uint64_t>(K) * 2, 64, 64))
    return cudaErrorInvalidValue;
  constexpr int CS = kClusterW;
  // x viewed as [K/64 chunks][M rows][64]: one box {64, 64 rows, 4/CS chunks} lands as
  // 8 KB 64x64 blocks, the MN-major layout of (a slice of) one operand entry
  int x3d = 0;
  if (K % 64 == 0) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(M), static_cast<uint64_t>(K / 64)};
    const uint64_t strides[2] = {static_cast<uint64_t>(K) * 2, 128};
    const uint32_t box[3] = {64, 64, 4 / CS};
    x3d = encode_tmap_3d_bf16(&mx3, x, dims, strides, box, 128) ? 1 : 0;
  }
  if (!x3d) mx3 = mx2;
  FusedArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.status = status_word_ptr();
  a.tiles_k = static_cast<int>((K + 511) / 512);
  a.dy = dy;
  a.g = g;
  a.fc = fc;
  a.dw_g = dw_g;
  a.dw_fc = dw_fc;
  a.ws = dw_part;
  a.db_part = db_part;
  a.splits = static_cast<int>(plan.splits);
  a.kb_per = static_cast<int>(plan.kb_per);
  a.nkb_total = static_cast<int>((M + 63) / 64);
  a.tiles_n = static_cast<int>(((N + 63) / 64 + CS - 1) / CS * CS);  // clusters of CS n tiles
  a.x3d = x3d;
  a.accumulate = accumulate ? 1 : 0;
  a.wait_limit = kWaitLimitCycles;
  a.stall_at = -1;
  const int64_t ctas = plan.splits * a.tiles_k * a.tiles_n;
  return launch<kFW, CS>(static_cast<unsigned>(ctas), stream, mdy, mg, mfc, mx3, mx2, mx2, a, false);
}

}  // namespace

cudaError_t launch_fused_w(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                           uint16_t* dw_g, uint16_t* dw_fc, uint16_t* db_g, uint16_t* db_fc, int64_t M, int64_t K,
                           int64_t N, void* ws, const FwPlan& plan, cudaStream_t stream, bool accumulate) {
  const size_t dw_bytes = plan.splits > 1 ? static_cast<size_t>(plan.splits) * 2 * K * N * sizeof(float) : 0;
  float* dw_part = static_cast<float*>(ws);
  float* db_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256(dw_bytes));
  cudaError_t e = launch_fw_kernel(x, dy, g, fc, dw_g, dw_fc, M, K, N, dw_part, db_part, plan, stream, accumulate);
  if (e != cudaSuccess) return e;
  if (plan.splits > 1) {
    e = launch_w_split_reduce(dw_part, plan.splits, K, N, dw_g, dw_fc, stream, accumulate);
    if (e != cudaSuccess) return e;
  }
  return launch_db_reduce(db_part, plan.splits, N, db_g, db_fc, stream, accumulate);
}

cudaError_t launch_fused_w_partials(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                                    int64_t M, int64_t K, int64_t N, float* dw_part, float* db_part,
                                    const FwPlan& plan, cudaStream_t stream) {
  if (plan.splits < 2) return cudaErrorInvalidValue;  // one split would write bf16 dw directly
  return launch_fw_kernel(x, dy, g, fc, nullptr, nullptr, M, K, N, dw_part, db_part, plan, stream, false);
}

}  // namespace swg
