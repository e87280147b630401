// Fused variant of the SwiGLU-FFN backward: the b-stage math runs inside the
// GEMMs' operand producer, so dg and dfc are formed tile by tile in shared
// memory and never written to (or read back from) HBM.
//
// Sources: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Algorithm overview and formulas" items 1-4 (the math of every stage); the
// recompute-instead-of-store principle stated in the Ascend C backward blog
// post (Swish section: recompute sigma in the backward rather than keep it).
//
// One CTA per SM: warpgroup 0 and the transform warps (FX: sixteen, FW: eight).
//   warp 0 lane 0   TMA producer of the operand ring (W chunks for FX, x chunks
//                   for FW; 128-byte swizzle)
//   warp 1          tensor-memory allocation (512 columns); lane 0 issues
//                   tcgen05.mma (K = 16) and tcgen05.commit (FW: in the pair's
//                   leader only)
//   warp 2 lane 0   L2 prefetch of the raw dy, g, fc tiles a few stages ahead
//                   of the transform, paced by the transform's progress count
//   warp 3          idle
//   warps 4-        transform: load dy, g, fc straight from global memory into
//                   registers (FX: two stages of registers, the loads running a
//                   stage ahead of the math; FW: three), compute dg, dfc in fp32
//                   and store them as bf16 into a ring of A-operand slots in the
//                   128-byte-swizzled layout the tensor core reads; then the
//                   epilogue.
// Warpgroup 0 gives registers to the transform warpgroups (setmaxnreg): 48 per
// thread there; FX's sixteen transform warps rise from the 96 a 640-thread
// block is launched with to 104, FW's eight from 168 to 224. Sixteen FX warps
// of two rows per stage with two register stages measured slightly faster than
// eight of four rows with three.
//
// fused x (FX): one CTA per MMA (M = 128, N = 256), persistent over m tiles.
//   D = dx[m0:m0+128, k0:k0+512] in two 256-column accumulator halves. Stages
//   of 64 reduction columns n. A = dg or dfc [128 m x 64 n] (K-major), B =
//   W_g / W_fc chunks [256 k x 64 n] (32 KB ring entries). A tile's epilogue
//   runs once the next tile's first stages are in their A slots, and it drains
//   the low accumulator half first and releases it, so the next tile's first
//   stages run their low-half MMAs while the high half is still being drained.
// fused w (FW): CTA pairs (clusters of 2); one tcgen05.mma.cta_group::2
//   (M = 256, N = 256) spans both SMs. Each CTA owns a 64-column band of n:
//   D = [dw_g^T ; dw_fc^T][n0:n0+64, k0:k0+512] in its own tensor memory, with
//   an A operand stacking 64 columns of dg over the same 64 columns of dfc
//   (MN-major; the two 8 KB halves of a slot are the two 64-element MN chunks,
//   LBO = 8 KB) that it forms itself. B = x [64 m x 256 k] per accumulator half
//   (MN-major), split along N: each CTA copies its 128 columns of k into its own
//   shared memory, one 32 KB ring entry per stage holding both halves, so every
//   SM streams half of x. The even CTA (the leader) issues the MMAs. One
//   barrier per stage slot (four slots, each an x entry and an A slot)
//   collects the stage's copies of both CTAs and the arrivals of both CTAs'
//   transform warps, and one release per stage is committed to the barriers of
//   both CTAs, so the leader checks one barrier per eight pair MMAs. Stages of
//   64 rows of m. Each CTA sums its dg, dfc columns over its rows in registers
//   (db column partials, one row per M split). The reduction over M is split
//   into S chunks with fp32 partials and a fixed-order reduce.
//
// Every mbarrier wait is bounded; a timeout sets the module status word,
// stops issuing, waits (bounded) for the work already issued, frees tensor
// memory and returns.
#include "swg_device.cuh"
#include "swg_launch.h"

namespace swg {

namespace {

enum FusedMode : int { kFX = 0, kFW = 1 };

constexpr int kXWarp0 = 4;      // first transform warp
constexpr int kCtlRegs = 48;    // registers per thread in warpgroup 0 after setmaxnreg
constexpr uint32_t kTmemCols = 512;
constexpr int kSplitStages = 2;  // FX: stages whose low-half MMAs run before the high half is free

template <int MODE>
struct Cfg;
template <>
struct Cfg<kFX> {
  static constexpr int kXWarps = 16;       // transform warps
  static constexpr int kThreads = 640;
  static constexpr int kLaunchRegs = 96;   // registers per thread at launch (65536 / 640, rounded down to 8)
  static constexpr int kXRegs = 104;       // transform warps after setmaxnreg
  static constexpr int kPair = 1;          // CTAs per MMA: single-CTA tcgen05.mma
  static constexpr int kRows = 128;        // m rows of a stage's tile (64 columns of n)
  static constexpr int kAStages = 3;       // A-operand slots (dg + dfc, 2 x 16 KB each)
  static constexpr int kEntryBytes = 32768;  // W_g or W_fc [256 k x 64 n]
  static constexpr int kEntries = 4;
  static constexpr int kPrefetch = 4;      // stages prefetched into L2 ahead of the loads
};
template <>
struct Cfg<kFW> {
  static constexpr int kXWarps = 8;
  static constexpr int kThreads = 384;
  static constexpr int kLaunchRegs = 168;
  static constexpr int kXRegs = 224;
  static constexpr int kPair = 2;          // CTAs per MMA: a cta_group::2 pair (M = 256)
  static constexpr int kRows = 64;         // m rows of a stage (64 columns of n)
  static constexpr int kAStages = 4;       // A-operand slots (dg | dfc stacked, 16 KB each)
  static constexpr int kEntryBytes = 65536 / kPair;  // x [64 m x 2 x 128 k]: this CTA's half of a stage
  static constexpr int kEntries = 4;       // = kAStages: entry i and A slot i form stage slot i
  static constexpr int kPrefetch = 4;
};

template <int MODE>
struct __align__(1024) FSmem {
  using C = Cfg<MODE>;
  static constexpr int kHalf = C::kRows * 128;  // one 64-column bf16 tile (dg or dfc)
  uint8_t ring[C::kEntries][C::kEntryBytes];
  uint8_t aop[C::kAStages][2 * kHalf];          // [dg | dfc]
  uint64_t a_full[C::kAStages];      // FX: the transform warps have written the slot
  uint64_t a_empty[C::kAStages];     // FX: the MMAs reading the slot are done
  uint64_t ring_full[C::kEntries];   // the entry's copies have landed (FW, leader: both CTAs'
                                     // halves, and both CTAs' transform warps wrote A slot i)
  uint64_t ring_empty[C::kEntries];  // the MMAs reading the entry (FW: and A slot i) are done
  uint64_t accum;                    // one phase per tile: the tile's MMAs are done
  uint64_t tmem_free[2];             // leader, one phase per tile per accumulator half: both
                                     // CTAs' epilogues have read it
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  volatile uint32_t ring_issued, ring_consumed;
  volatile uint32_t x_progress;      // stages the transform has produced (paces the prefetch warp)
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
  int tile0;          // FX: the first m tile of this launch (tiles tile0 + ct)
  int cluster_tiles;  // pair tiles; cluster c takes c, c + nclusters, ...
  int accumulate;     // FW: dw, db += this call's sums (one rounding of old + new)
  long long wait_limit;  // cycles before a pipeline wait gives up
  int64_t stall_at;      // test injection: the producer stops before this ring entry (-1: never)
};

// One CTA's share of one pair tile.
struct Tile {
  int m0, n0, k0, kt, split, nst, kb_begin, nh, eps;
};

template <int MODE>
__device__ __forceinline__ Tile tile_of(int ct, uint32_t crank, const FusedArgs& args) {
  constexpr int kPair = Cfg<MODE>::kPair;
  Tile t;
  t.m0 = t.n0 = t.split = t.kb_begin = 0;
  if (MODE == kFX) {
    // a 128-row m tile at one 512-column block of K
    static_assert(Cfg<kFX>::kPair == 1, "FX runs on single-CTA MMAs");
    const int c2 = ct + args.tile0;
    t.kt = c2 % args.tiles_k;
    t.m0 = (c2 / args.tiles_k) * 128;
    t.nst = (args.N + 63) / 64;  // stages: 64 columns of n each
  } else {
    // pair tile = 2 consecutive 64-column bands of n, one K block, one M split
    const int bands = args.tiles_n / kPair;
    t.n0 = ((ct % bands) * kPair + static_cast<int>(crank)) * 64;
    const int rest = ct / bands;
    t.kt = rest % args.tiles_k;
    t.split = rest / args.tiles_k;
    t.kb_begin = t.split * args.kb_per;
    t.nst = min(args.nkb_total, t.kb_begin + args.kb_per) - t.kb_begin;  // stages: 64 rows of m each
  }
  t.k0 = t.kt * 512;
  t.nh = (args.K - t.k0) > 256 ? 2 : 1;             // 256-column accumulator halves in use
  t.eps = (MODE == kFX) ? 2 * t.nh : 1;             // ring entries per stage
  return t;
}

// FX entry order within a tile: the first J stages issue their low-half (h = 0)
// entries first, then their high-half entries, so that their low-half MMAs can
// run while the previous tile's high accumulator half is still being drained.
struct EntryPos {
  int i, p, h;
};
__device__ __forceinline__ EntryPos fx_entry(const Tile& tl, int j) {
  const int J = tl.nh == 2 ? min(kSplitStages, tl.nst) : 0;
  EntryPos r;
  if (j < 2 * J) {
    r.i = j >> 1;
    r.p = j & 1;
    r.h = 0;
  } else if (j < 4 * J) {
    r.i = (j - 2 * J) >> 1;
    r.p = j & 1;
    r.h = 1;
  } else {
    const int jj = j - 4 * J;
    r.i = J + jj / tl.eps;
    const int q = jj % tl.eps;
    r.p = q / tl.nh;
    r.h = q % tl.nh;
  }
  return r;
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
template <int XW>
__device__ __forceinline__ void named_sync_transform() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * XW) : "memory");
}

// has the phase with the given parity completed? (a non-blocking look)
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
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

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::kThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_g,
                 const __grid_constant__ CUtensorMap tm_fc, const __grid_constant__ CUtensorMap tm_b0,
                 const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_out,
                 const FusedArgs args) {
  using S = FSmem<MODE>;
  using C = Cfg<MODE>;
  constexpr int kPair = C::kPair;
  constexpr int kAS = C::kAStages;
  constexpr int kRE = C::kEntries;
  constexpr int kRows = C::kRows;
  constexpr int kHalf = S::kHalf;
  constexpr int kXWarps = C::kXWarps;
  constexpr int kRS = kXWarps * 4;     // row stride: transform threads per 8-column chunk
  constexpr int kRPT = kRows / kRS;    // rows per transform thread per stage
  extern __shared__ uint8_t smem_raw[];
  S& s = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t crank = kPair == 2 ? cluster_ctarank() : 0u;  // rank in the pair (FX: no cluster)
  const bool leader = crank == 0;
  const int cluster = blockIdx.x / kPair;
  const int nclusters = gridDim.x / kPair;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAS; ++i) {
      mbar_init(&s.a_full[i], kPair * kXWarps);
      mbar_init(&s.a_empty[i], 1);
    }
    for (int i = 0; i < kRE; ++i) {
      // FW: the stage's x copies and both CTAs' A slots complete one barrier
      mbar_init(&s.ring_full[i], MODE == kFW ? 1 + kPair * kXWarps : 1);
      mbar_init(&s.ring_empty[i], 1);
    }
    mbar_init(&s.accum, 1);
    mbar_init(&s.tmem_free[0], kPair * kXWarps);
    mbar_init(&s.tmem_free[1], kPair * kXWarps);
    s.abort_flag = 0u;
    s.ring_issued = s.ring_consumed = 0u;
    s.x_progress = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_dy);
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_fc);
    tma_prefetch_desc(&tm_b0);
    tma_prefetch_desc(&tm_b1);
  }
  if (warp == 1) {
    if (kPair == 2) {
      tmem_alloc_pair(&s.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&s.tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (kPair == 2) cluster_sync();  // both CTAs' barriers are initialised before any remote arrival or copy
  const uint32_t tmem = s.tmem_base;

  if (warp < kXWarp0) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs) : "memory");
  static_assert(kRows % kRS == 0, "rows per transform thread");

  if (warp == 0) {
    // ------------------------------------------------------------ operand producer (both CTAs)
    if (lane == 0) {
      uint32_t gj = 0;  // ring entries issued, over all tiles
      bool stopped = false;
      for (int ct = cluster; ct < args.cluster_tiles && !s.abort_flag && !stopped; ct += nclusters) {
        const Tile tl = tile_of<MODE>(ct, crank, args);
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
          // the leader's barrier counts both halves of the entry
          if (leader) mbar_arrive_expect_tx(&s.ring_full[e], MODE == kFX ? kPair * C::kEntryBytes : tl.nh * 32768u);
          const uint32_t full = kPair == 2 ? cluster_addr(&s.ring_full[e], 0) : 0u;
          if (MODE == kFX) {
            const EntryPos ep = fx_entry(tl, j);
            const int kr = tl.k0 + 256 * ep.h + (256 / kPair) * static_cast<int>(crank);
            if (kPair == 2)
              tma_load_2d_pair(s.ring[e], ep.p ? &tm_b1 : &tm_b0, full, ep.i * 64, kr);
            else
              tma_load_2d(s.ring[e], ep.p ? &tm_b1 : &tm_b0, &s.ring_full[e], ep.i * 64, kr);
          } else {
            const int mrow = (tl.kb_begin + j) * 64;
            for (int h = 0; h < tl.nh; ++h) {
              const int kk = tl.k0 + 256 * h + (256 / kPair) * static_cast<int>(crank);
              uint8_t* dst = s.ring[e] + h * (32768 / kPair);
#pragma unroll
              for (int cbox = 0; cbox < 4 / kPair; ++cbox) {
                if (kPair == 2)
                  tma_load_2d_pair(dst + cbox * 8192, &tm_b0, full, kk + 64 * cbox, mrow);
                else
                  tma_load_2d(dst + cbox * 8192, &tm_b0, &s.ring_full[e], kk + 64 * cbox, mrow);
              }
            }
          }
          s.ring_issued = gj + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(128 * kPair, 256, MODE == kFW, MODE == kFW);
      uint32_t gi = 0, gj = 0, tt = 0;  // A stages, ring entries, tiles consumed
      bool ok = true;
      // a release goes to the barrier at the same offset in both CTAs
      auto commit2 = [&](uint64_t* bar) {
        if (kPair == 2) {
          umma_commit_pair(cluster_addr(bar, 0));
          umma_commit_pair(cluster_addr(bar, 1));
        } else {
          umma_commit(bar);
        }
      };
      auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t acc) {
        if (kPair == 2)
          umma_pair(d, ad, bd, idesc, acc);
        else
          umma_bf16(d, ad, bd, idesc, acc);
      };
      auto consume = [&](int i, int p, int h) -> bool {
        const int e = gj % kRE;
        if (!mbar_wait(&s.ring_full[e], (gj / kRE) & 1, args.wait_limit)) {
          flag_timeout(s, args.status);
          return false;
        }
        s.ring_consumed = gj + 1;
        tc_fence_after();
        const uint32_t b_addr = smem_u32(s.ring[e]);
        const uint32_t a_slot = smem_u32(s.aop[(gi + i) % kAS]);
        if (MODE == kFX) {
          const uint32_t a_addr = a_slot + p * kHalf;  // dg or dfc
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma(tmem + h * 256, smem_desc(a_addr + 32 * k, 16, 1024), smem_desc(b_addr + 32 * k, 16, 1024),
                (i > 0 || p > 0 || k > 0) ? 1u : 0u);
        } else {
          for (int hh = 0; hh < h; ++hh)  // h: the halves in use
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + hh * 256, smem_desc(a_slot + 2048 * k, kHalf, 1024),
                  smem_desc(b_addr + hh * (32768 / kPair) + 2048 * k, 8192, 1024), (i > 0 || k > 0) ? 1u : 0u);
        }
        commit2(&s.ring_empty[e]);
        ++gj;
        return true;
      };
      auto wait_a = [&](int i) -> bool {
        const uint32_t g2 = gi + i;
        if (!mbar_wait(&s.a_full[g2 % kAS], (g2 / kAS) & 1, args.wait_limit)) {
          flag_timeout(s, args.status);
          return false;
        }
        tc_fence_after();
        return true;
      };
      // the previous tile's epilogue has read accumulator half h out
      auto wait_free = [&](int h) -> bool {
        if (tt == 0) return true;
        if (!mbar_wait(&s.tmem_free[h], (tt - 1) & 1, args.wait_limit)) {
          flag_timeout(s, args.status);
          return false;
        }
        tc_fence_after();
        return true;
      };
      for (int ct = cluster; ct < args.cluster_tiles && ok; ct += nclusters, ++tt) {
        const Tile tl = tile_of<MODE>(ct, 0u, args);
        if (MODE == kFX) {
          // the first J stages: low-half MMAs as soon as the low half is free, then
          // their high-half MMAs once the high half is free too
          const int J = tl.nh == 2 ? min(kSplitStages, tl.nst) : 0;
          if (!wait_free(0)) break;
          if (J == 0 && !wait_free(1)) break;
          for (int i = 0; i < J && ok; ++i) {
            ok = wait_a(i);
            for (int p = 0; p < 2 && ok; ++p) ok = consume(i, p, 0);
          }
          if (ok && J > 0) ok = wait_free(1);
          for (int i = 0; i < J && ok; ++i) {
            for (int p = 0; p < 2 && ok; ++p) ok = consume(i, p, 1);
            commit2(&s.a_empty[(gi + i) % kAS]);
          }
          for (int i = J; i < tl.nst && ok; ++i) {
            ok = wait_a(i);
            for (int q = 0; q < tl.eps && ok; ++q) ok = consume(i, q / tl.nh, q % tl.nh);
            commit2(&s.a_empty[(gi + i) % kAS]);
          }
        } else {
          if (!wait_free(0) || !wait_free(1)) break;
          for (int i = 0; i < tl.nst && ok; ++i) {
            ok = consume(i, 0, tl.nh);
          }
        }
        gi += tl.nst;
        commit2(&s.accum);  // this tile's accumulators (both CTAs) are complete
      }
      // after a timeout the epilogues may have stopped waiting: see every MMA this thread
      // issued complete before tensor memory is freed (tt accumulator phases were committed)
      if (s.abort_flag && tt > 0) mbar_wait(&s.accum, (tt - 1) & 1, args.wait_limit);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ L2 prefetch of the raw tiles
    if (lane == 0) {
      int ntot = 0;
      for (int ct = cluster; ct < args.cluster_tiles; ct += nclusters) ntot += tile_of<MODE>(ct, crank, args).nst;
      int next = 0, tix = 0, in_tile = 0;
      Tile tl = tile_of<MODE>(cluster, crank, args);
      uint32_t last = 0;
      long long tlast = clock64();
      while (next < ntot && !s.abort_flag) {
        const uint32_t pr = s.x_progress;
        if (pr != last) {
          last = pr;
          tlast = clock64();
        }
        if (next < static_cast<int>(pr) + C::kPrefetch + 1) {
          if (MODE == kFX) {
            const int p0 = in_tile * 64;
            tma_prefetch_l2_2d(&tm_dy, p0, tl.m0);
            tma_prefetch_l2_2d(&tm_g, p0, tl.m0);
            tma_prefetch_l2_2d(&tm_fc, p0, tl.m0);
          } else {
            const int p1 = (tl.kb_begin + in_tile) * 64;
            tma_prefetch_l2_2d(&tm_dy, tl.n0, p1);
            tma_prefetch_l2_2d(&tm_g, tl.n0, p1);
            tma_prefetch_l2_2d(&tm_fc, tl.n0, p1);
          }
          ++next;
          if (++in_tile == tl.nst) {
            in_tile = 0;
            ++tix;
            tl = tile_of<MODE>(cluster + tix * nclusters, crank, args);
          }
        } else {
          if (clock64() - tlast > args.wait_limit) break;  // the transform stopped making progress
          __nanosleep(64);
        }
      }
    }
  } else if (warp >= kXWarp0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kXRegs) : "memory");
    // ------------------------------------------------------------ transform (both CTAs)
    const int t = threadIdx.x - kXWarp0 * 32;  // 0 .. 32 kXWarps - 1
    const int xw = warp - kXWarp0;             // transform warp
    const int c = t & 7;                       // 16-byte chunk of the 64-column tile (8 columns)
    const int rg = t >> 3;                     // row group; rows rg, rg + kRS, ...
    const int64_t N64 = args.N;
    // A thread whose wait runs out stops computing ("dead") but keeps taking
    // part in the arrivals and the named barriers.
    bool dead = false;

    // arrival of this warp on a barrier of the pair leader (after its lanes' work)
    auto warp_arrive_leader = [&](uint64_t* bar, bool may = true) {
      __syncwarp();
      if (lane == 0 && may) {
        if (kPair == 1 || leader)
          mbar_arrive(bar);
        else
          mbar_arrive_remote(cluster_addr(bar, 0));
      }
    };
    // stores one stage's dg, dfc (8 columns x kRPT rows of this thread) into A slot a
    auto store_stage = [&](int a, int row0, int col, bool want_dg, const uint4 (&bdy)[kRPT],
                           const uint4 (&bg)[kRPT], const uint4 (&bfc)[kRPT], float (&cg)[8], float (&cf)[8]) {
      const uint32_t sdg = smem_u32(s.aop[a]);
      const uint32_t sdf = sdg + kHalf;
#pragma unroll
      for (int q = 0; q < kRPT; ++q) {
        const int row = rg + kRS * q;  // row within the tile
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
        const int row = row0 + rg + kRS * q;
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
      uint64_t* eb = MODE == kFW ? &s.ring_empty[a] : &s.a_empty[a];
      if (!dead && st >= kAS && !mbar_wait(eb, ((st / kAS) - 1) & 1, args.wait_limit)) {
        flag_timeout(s, args.status);
        dead = true;
      }
      if (s.abort_flag) dead = true;
    };
    uint4 xdy[kRPT], xg[kRPT], xfc[kRPT], ydy[kRPT], yg[kRPT], yfc[kRPT], zdy[kRPT], zg[kRPT], zfc[kRPT];

    if constexpr (MODE == kFX) {
      // The CTA's stages form one stream over its tiles: stage st is stage
      // st % nst of the CTA's tile st / nst, and also the global A-stage index.
      // A tile's epilogue runs after the first kAS - 1 stages of the next tile
      // are in their A slots; the staging buffer of the epilogue's TMA stores
      // is the A slot of the finished tile's last stage, free once its MMAs are.
      const int nst = (args.N + 63) / 64;
      const int ntiles = cluster < args.cluster_tiles ? (args.cluster_tiles - 1 - cluster) / nclusters + 1 : 0;
      const int total = ntiles * nst;
      const int look = nst < kAS - 1 ? nst : kAS - 1;
      auto tile_at = [&](int tix) { return tile_of<MODE>(cluster + tix * nclusters, crank, args); };
      float ug[8], uf[8];  // column sums, unused here
#pragma unroll
      for (int e = 0; e < 8; ++e) ug[e] = uf[e] = 0.0f;

      // a position in the CTA's stage stream: stage index, stage within its tile, tile index,
      // and the tile's first row and K block, advanced without divisions
      struct Cur {
        int st, sit, tix, m0, kt;
      };
      auto advance = [&](Cur& p) {
        ++p.st;
        if (++p.sit == nst) {
          p.sit = 0;
          ++p.tix;
          if (p.st < total) {
            const Tile tl = tile_at(p.tix);
            p.m0 = tl.m0;
            p.kt = tl.kt;
          }
        }
      };
      const Tile tl0 = tile_at(0);
      Cur lc{0, 0, 0, tl0.m0, tl0.kt};  // the next stage to load
      Cur pc = lc;                       // the next stage to transform
      auto load = [&](uint4 (&bdy)[kRPT], uint4 (&bg)[kRPT], uint4 (&bfc)[kRPT]) {
        const bool valid = lc.st < total;
        load_rows(valid ? lc.m0 : 0, (valid ? lc.sit * 64 : 0) + c * 8, valid, bdy, bg, bfc);
        advance(lc);
      };
      auto process = [&](const uint4 (&bdy)[kRPT], const uint4 (&bg)[kRPT], const uint4 (&bfc)[kRPT]) {
        const int st = pc.st;
        const int a = st % kAS;
        acquire_slot(static_cast<uint32_t>(st), a);
        if (!dead)
          store_stage(a, pc.m0, pc.sit * 64 + c * 8, pc.kt == 0 && args.dg_out != nullptr, bdy, bg, bfc, ug, uf);
        warp_arrive_leader(&s.a_full[a]);
        if (t == 0) s.x_progress = static_cast<uint32_t>(st + 1);
      };
      // tile tix's accumulator -> bf16 dx through staging buffer stg (an A slot):
      // the low half (columns 0-255) first, then the high half, each released to the
      // leader as soon as it has been read
      auto epilogue = [&](int tix, int stg) {
        const Tile tl = tile_at(tix);
        bool acc_ok = false;
        if (!dead && !s.abort_flag) {
          acc_ok = mbar_wait(&s.accum, tix & 1, args.wait_limit);
          if (!acc_ok) flag_timeout(s, args.status);
        }
        const int q = warp & 3;    // TMEM lane quarter this warp may read
        // the warps of a lane quarter split each 256-column accumulator half into kSubW-column parts
        constexpr int kSubW = 256 / (kXWarps / 4);
        constexpr int kStgBufs = (2 * kHalf / kXWarps) / 2048;  // 2 KB staging blocks per warp
        static_assert(kStgBufs >= 1, "staging");
        const int sub = xw >> 2;
        tc_fence_after();
        // tcgen05.ld is warp-collective: decide for the whole warp
        const bool go = __all_sync(0xffffffffu, !dead && acc_ok && !s.abort_flag);
        int nb = 0;  // blocks stored by this warp (alternating 2 KB staging halves)
        for (int h = 0; h < 2; ++h) {
          if (go && h < tl.nh) {
#pragma unroll 1
            for (int cc = 0; cc < kSubW / 32; ++cc, ++nb) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 256 + sub * kSubW + cc * 32, v);
              tmem_ld_wait();
              // this warp's 32 x 32 block -> a 64-byte-swizzled staging buffer -> one TMA
              // store (rows beyond M and columns beyond K are clipped by the copy engine)
              uint8_t* buf = s.aop[stg] + xw * (2048 * kStgBufs) + (nb % kStgBufs) * 2048;
              if (nb >= kStgBufs) {
                if (lane == 0) bulk_wait_read<kStgBufs - 1>();  // the store that used this buffer has read it
                __syncwarp();
              }
              const uint32_t sb = smem_u32(buf) + lane * 64;
#pragma unroll
              for (int j = 0; j < 4; ++j) sts128(sb + ((j ^ ((lane >> 1) & 3)) << 4), pack8(v + 8 * j));
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tm_out, buf, tl.k0 + h * 256 + sub * kSubW + cc * 32, tl.m0 + q * 32);
                bulk_commit();
              }
            }
          }
          tc_fence_before();
          warp_arrive_leader(&s.tmem_free[h]);  // this warp has read its part of half h
        }
        // the staging slot is written again by a later stage: every store has read it
        if (lane == 0) bulk_wait_read<0>();
        named_sync_transform<kXWarps>();
      };
      auto after = [&]() {
        if (pc.tix >= 1 && pc.sit + 1 == look) epilogue(pc.tix - 1, (pc.tix * nst - 1) % kAS);
        advance(pc);
      };

      // two stages of registers: the loads of stage st + 1 are in flight while stage
      // st is computed (and while an epilogue runs)
      load(xdy, xg, xfc);
      for (int st = 0; st < total; st += 2) {
        load(ydy, yg, yfc);
        process(xdy, xg, xfc);
        after();
        if (st + 1 >= total) break;
        load(xdy, xg, xfc);
        process(ydy, yg, yfc);
        after();
      }
      if (ntiles > 0) epilogue(ntiles - 1, (total - 1) % kAS);
      if (lane == 0) bulk_wait_all();  // every store has landed before the CTA exits
    } else {
      uint32_t gi = 0, tt = 0;  // A stages, tiles produced
      for (int ct = cluster; ct < args.cluster_tiles; ct += nclusters, ++tt) {
        const Tile tl = tile_of<MODE>(ct, crank, args);
        const int n0 = tl.n0, k0 = tl.k0, kb_begin = tl.kb_begin, nst = tl.nst, nh = tl.nh, split = tl.split;
        const bool want_db = tl.kt == 0 && args.db_part != nullptr;
        float cg[8], cf[8];  // column sums over the CTA's whole M range
#pragma unroll
        for (int e = 0; e < 8; ++e) cg[e] = cf[e] = 0.0f;

        auto load = [&](int i, uint4 (&bdy)[kRPT], uint4 (&bg)[kRPT], uint4 (&bfc)[kRPT]) {
          load_rows((kb_begin + i) * 64, n0 + c * 8, i < nst, bdy, bg, bfc);
        };
        auto process = [&](int i, const uint4 (&bdy)[kRPT], const uint4 (&bg)[kRPT], const uint4 (&bfc)[kRPT]) {
          const uint32_t gs = gi + i;  // global A-stage index
          const int a = gs % kAS;
          acquire_slot(gs, a);
          if (!dead) store_stage(a, (kb_begin + i) * 64, n0 + c * 8, false, bdy, bg, bfc, cg, cf);
          // The slot's barrier also counts the producer's copies. A warp whose wait ran out (lane 0
          // decides) arrives only where the slot's previous use was released: that use's phase
          // completed, so this arrival falls into the phase of stage gs, and an arrival can never
          // overrun a phase that a missing copy left open.
          const bool may = lane != 0 || !dead || gs < static_cast<uint32_t>(kAS) ||
                           mbar_test(smem_u32(&s.ring_empty[a]), ((gs / kAS) - 1) & 1);
          warp_arrive_leader(&s.ring_full[a], may);
          if (t == 0) s.x_progress = gs + 1;
        };

        load(0, xdy, xg, xfc);
        load(1, ydy, yg, yfc);
        for (int i = 0; i < nst; i += 3) {
          load(i + 2, zdy, zg, zfc);
          process(i, xdy, xg, xfc);
          if (i + 1 >= nst) break;
          load(i + 3, xdy, xg, xfc);
          process(i + 1, ydy, yg, yfc);
          if (i + 2 >= nst) break;
          load(i + 4, ydy, yg, yfc);
          process(i + 2, zdy, zg, zfc);
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
          named_sync_transform<kXWarps>();
          float* scratch = reinterpret_cast<float*>(s.aop[0]);  // [8 warps][8 chunks][16]
          if (lane < 8) {
            float* pp = scratch + (xw * 8 + c) * 16;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              pp[e] = cg[e];
              pp[8 + e] = cf[e];
            }
          }
          named_sync_transform<kXWarps>();
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
          named_sync_transform<kXWarps>();  // the scratch is read before a later tile's stage reuses the slot
        }

        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        tc_fence_after();
        const int r = q * 32 + lane;    // accumulator row (TMEM lane)
        const int h = xw >> 2;          // accumulator half this warp drains
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
        warp_arrive_leader(&s.tmem_free[0]);  // this warp has read its part of the accumulator
        warp_arrive_leader(&s.tmem_free[1]);
      }  // tile loop
    }
  }

  __syncthreads();
  if (kPair == 2) cluster_sync();  // both CTAs are done with their roles: no more remote arrivals or commits
  if (leader && threadIdx.x == 0) {
    const uint32_t peer_abort = kPair == 2 ? ld_cluster_u32(&s.abort_flag, 1) : 0u;
    if (s.abort_flag || peer_abort) {
      // drain: copies (of either CTA) that complete on this CTA's barriers must land
      // before any CTA exits
      const uint32_t peer_issued = kPair == 2 ? ld_cluster_u32(&s.ring_issued, 1) : 0u;
      const uint32_t issued = s.ring_issued > peer_issued ? s.ring_issued : peer_issued;
      for (uint32_t i = s.ring_consumed; i < issued; ++i)
        if (!mbar_wait(&s.ring_full[i % kRE], (i / kRE) & 1, args.wait_limit)) break;
    }
  }
  if (kPair == 2) cluster_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (kPair == 2)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE>
constexpr size_t smem_bytes() {
  return sizeof(FSmem<MODE>) + 1024;
}

template <int MODE>
cudaError_t launch(unsigned grid, cudaStream_t stream, const CUtensorMap& a, const CUtensorMap& b,
                   const CUtensorMap& c, const CUtensorMap& d, const CUtensorMap& e, const CUtensorMap& out,
                   FusedArgs args, bool persistent, int max_ctas = 0) {
  constexpr int kPair = Cfg<MODE>::kPair;
  constexpr size_t smem = smem_bytes<MODE>();
  static_assert(MODE == kFX || Cfg<kFW>::kEntries == Cfg<kFW>::kAStages, "fw slots");
  static_assert(smem <= 232448, "fused kernel shared memory");
  using C = Cfg<MODE>;
  constexpr int kThreads = C::kThreads;
  static_assert(128 * kCtlRegs + (kThreads - 128) * C::kXRegs <= kThreads * C::kLaunchRegs,
                "setmaxnreg split exceeds the launch's registers");
  cudaError_t err = cudaFuncSetAttribute(fused_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  {
    // setmaxnreg redistributes the block's launch registers: warpgroup 0 drops to
    // kCtlRegs per thread, the two transform warpgroups rise to kXRegs. The sum must
    // fit what the block was launched with, else an increase would wait forever:
    // refuse to launch otherwise.
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, fused_kernel<MODE>);
    if (err != cudaSuccess) return err;
    if (static_cast<long long>(fa.numRegs) * kThreads < 128LL * kCtlRegs + (kThreads - 128LL) * C::kXRegs)
      return cudaErrorInvalidValue;
  }
  args.cluster_tiles = static_cast<int>(grid / kPair);
  if constexpr (kPair == 1) {
    if (persistent) {
      // one resident wave, each CTA looping over tiles
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel<MODE>, kThreads, smem) ==
              cudaSuccess &&
          per_sm > 0) {
        const unsigned wave = static_cast<unsigned>(per_sm * device_sm_count());
        if (wave < grid) grid = wave;
      }
    }
    if (max_ctas > 0 && grid > static_cast<unsigned>(max_ctas)) grid = static_cast<unsigned>(max_ctas);
    fused_kernel<MODE><<<grid, kThreads, smem, stream>>>(a, b, c, d, e, out, args);
    return cudaGetLastError();
  } else {
    // clusters of two CTAs: the pair that one cta_group::2 MMA spans
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (persistent) {
      // one resident wave of pairs, each looping over pair tiles
      int max_clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&max_clusters, fused_kernel<MODE>, &cfg) == cudaSuccess &&
          max_clusters > 0 && static_cast<unsigned>(max_clusters) * kPair < grid)
        cfg.gridDim = dim3(static_cast<unsigned>(max_clusters) * kPair);
    }
    return cudaLaunchKernelEx(&cfg, fused_kernel<MODE>, a, b, c, d, e, out, args);
  }
}

inline size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

// The w stage's two reductions in one launch. Blocks [0, dw_blocks) add the dw split partials
// ws[s][p][k][n] in split order in fp32 and round once to bf16 (with accumulate, the old dw value
// joins the fp32 sum before the rounding); the other blocks add the db partials db_part[s][2N] in
// fp64 -- per column the splits s = r, r + 32, ... summed for each r < 32, those 32 sums then added
// in order -- and round once to bf16. The same arithmetic as the separate dw and db reduces.
// At most 32 registers a thread: a 64-thread block then fits on an SM beside a CTA of the fused x
// stage (640 threads of 96 registers leave 1024 registers on each SM sub-partition).
__global__ void __launch_bounds__(256, 8) fw_reduce_kernel(const float4* __restrict__ ws, int splits,
                                                        int64_t per_prob4, uint2* __restrict__ dw_g,
                                                        uint2* __restrict__ dw_fc, const float* __restrict__ db_part,
                                                        int64_t N, uint16_t* __restrict__ db_g,
                                                        uint16_t* __restrict__ db_fc, int accumulate,
                                                        int dw_blocks) {
  if (static_cast<int>(blockIdx.x) < dw_blocks) {
    const int64_t total4 = 2 * per_prob4;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total4;
         i += static_cast<int64_t>(dw_blocks) * blockDim.x) {
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
    return;
  }
  const int64_t two_n = 2 * N;
  const int64_t j = static_cast<int64_t>(static_cast<int>(blockIdx.x) - dw_blocks) * blockDim.x + threadIdx.x;
  if (j >= two_n) return;
  double t = 0.0;
  for (int r = 0; r < 32 && r < splits; ++r) {
    double sr = 0.0;
    for (int sp = r; sp < splits; sp += 32) sr += static_cast<double>(db_part[static_cast<int64_t>(sp) * two_n + j]);
    t += sr;
  }
  uint16_t* dst = j < N ? db_g + j : db_fc + (j - N);
  if (accumulate) t += static_cast<double>(__uint_as_float(static_cast<uint32_t>(*dst) << 16));
  const __nv_bfloat16 b = __double2bfloat16(t);
  *dst = *reinterpret_cast<const uint16_t*>(&b);
}

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
                           int64_t N, cudaStream_t stream, int64_t tile_begin, int64_t tile_end, int max_ctas) {
  CUtensorMap mdy, mg, mfc, mw0, mw1, mdx;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  if (!encode_tmap_2d_bf16(&mdx, dx, K, M, static_cast<uint64_t>(K) * 2, 32, 32, 64)) return cudaErrorInvalidValue;
  // the raw tensors are only prefetched into L2 here, one stage's box at a time
  if (!encode_tmap_2d_bf16(&mdy, dy, N, M, rs, 64, 128, 0) || !encode_tmap_2d_bf16(&mg, g, N, M, rs, 64, 128, 0) ||
      !encode_tmap_2d_bf16(&mfc, fc, N, M, rs, 64, 128, 0) ||
      !encode_tmap_2d_bf16(&mw0, w_g, N, K, rs, 64, 256) || !encode_tmap_2d_bf16(&mw1, w_fc, N, K, rs, 64, 256))
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
  const int64_t tiles = fused_x_tiles(M, K);
  if (tile_end < 0 || tile_end > tiles) tile_end = tiles;
  if (tile_begin < 0 || tile_begin >= tile_end) return cudaSuccess;  // nothing in the range
  a.tile0 = static_cast<int>(tile_begin);
  return launch<kFX>(static_cast<unsigned>(tile_end - tile_begin), stream, mdy, mg, mfc, mw0, mw1, mdx, a, true,
                     max_ctas);
}

int64_t fused_x_tiles(int64_t M, int64_t K) { return (M + 127) / 128 * ((K + 511) / 512); }

int64_t fused_w_ctas(int64_t K, int64_t N, const FwPlan& plan) {
  constexpr int kPair = Cfg<kFW>::kPair;
  return plan.splits * ((K + 511) / 512) * (((N + 63) / 64 + kPair - 1) / kPair * kPair);
}

namespace {

// the FW kernel alone: fp32 split partials into dw_part / db_part when plan.splits > 1, else bf16 dw
// straight into dw_g, dw_fc (db always as partials)
cudaError_t launch_fw_kernel(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                             uint16_t* dw_g, uint16_t* dw_fc, int64_t M, int64_t K, int64_t N, float* dw_part,
                             float* db_part, const FwPlan& plan, cudaStream_t stream, bool accumulate) {
  constexpr int kPair = Cfg<kFW>::kPair;
  CUtensorMap mdy, mg, mfc, mx;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  // x as 64 x 64 boxes (64 columns of k, 64 rows of m): 8 KB MN-major chunks
  if (!encode_tmap_2d_bf16(&mdy, dy, N, M, rs, 64, 64) || !encode_tmap_2d_bf16(&mg, g, N, M, rs, 64, 64) ||
      !encode_tmap_2d_bf16(&mfc, fc, N, M, rs, 64, 64) ||
      !encode_tmap_2d_bf16(&mx, x, K, M, static_cast<uint64_t>(K) * 2, 64, 64))
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
  a.dw_g = dw_g;
  a.dw_fc = dw_fc;
  a.ws = dw_part;
  a.db_part = db_part;
  a.splits = static_cast<int>(plan.splits);
  a.kb_per = static_cast<int>(plan.kb_per);
  a.nkb_total = static_cast<int>((M + 63) / 64);
  a.tiles_n = static_cast<int>(((N + 63) / 64 + kPair - 1) / kPair * kPair);  // pairs of 64-column bands
  a.accumulate = accumulate ? 1 : 0;
  const Injection inj = take_injection(3);
  a.wait_limit = inj.wait_limit;
  a.stall_at = inj.stall_at;
  const int64_t ctas = plan.splits * a.tiles_k * a.tiles_n;
  return launch<kFW>(static_cast<unsigned>(ctas), stream, mdy, mg, mfc, mx, mx, mx, a, false);
}

}  // namespace

namespace {
void fw_parts(void* ws, const FwPlan& plan, int64_t K, int64_t N, float** dw_part, float** db_part) {
  const size_t dw_bytes = plan.splits > 1 ? static_cast<size_t>(plan.splits) * 2 * K * N * sizeof(float) : 0;
  *dw_part = static_cast<float*>(ws);
  *db_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256(dw_bytes));
}
}  // namespace

cudaError_t launch_fused_w_kernel(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                                  uint16_t* dw_g, uint16_t* dw_fc, int64_t M, int64_t K, int64_t N, void* ws,
                                  const FwPlan& plan, cudaStream_t stream, bool accumulate) {
  float *dw_part, *db_part;
  fw_parts(ws, plan, K, N, &dw_part, &db_part);
  return launch_fw_kernel(x, dy, g, fc, dw_g, dw_fc, M, K, N, dw_part, db_part, plan, stream, accumulate);
}

cudaError_t launch_fused_w_reduce(void* ws, const FwPlan& plan, int64_t K, int64_t N, uint16_t* dw_g,
                                  uint16_t* dw_fc, uint16_t* db_g, uint16_t* db_fc, cudaStream_t stream,
                                  bool accumulate, int beside_ctas) {
  float *dw_part, *db_part;
  fw_parts(ws, plan, K, N, &dw_part, &db_part);
  const int64_t per_prob4 = K * N / 4;
  // beside_ctas > 0: at most that many blocks of 64 threads (32 registers each, no shared memory), so that
  // one fits on an SM beside a CTA of the x stage's persistent wave; the grid-stride loop takes the rest
  int threads = 256;
  int64_t cap = 4096;
  if (beside_ctas > 0 && (2 * N + 63) / 64 < beside_ctas) {
    threads = 64;
    cap = beside_ctas - (2 * N + 63) / 64;
  }
  int64_t dw_blocks = plan.splits > 1 ? (2 * per_prob4 + threads - 1) / threads : 0;
  if (dw_blocks > cap) dw_blocks = cap;
  const int64_t db_blocks = (2 * N + threads - 1) / threads;
  fw_reduce_kernel<<<static_cast<unsigned>(dw_blocks + db_blocks), static_cast<unsigned>(threads), 0, stream>>>(
      reinterpret_cast<const float4*>(dw_part), static_cast<int>(plan.splits), per_prob4,
      reinterpret_cast<uint2*>(dw_g), reinterpret_cast<uint2*>(dw_fc), db_part, N, db_g, db_fc, accumulate ? 1 : 0,
      static_cast<int>(dw_blocks));
  return cudaGetLastError();
}

cudaError_t launch_fused_w(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                           uint16_t* dw_g, uint16_t* dw_fc, uint16_t* db_g, uint16_t* db_fc, int64_t M, int64_t K,
                           int64_t N, void* ws, const FwPlan& plan, cudaStream_t stream, bool accumulate) {
  cudaError_t e = launch_fused_w_kernel(x, dy, g, fc, dw_g, dw_fc, M, K, N, ws, plan, stream, accumulate);
  if (e != cudaSuccess) return e;
  // both reductions in one launch (with one split the kernel wrote dw itself)
  return launch_fused_w_reduce(ws, plan, K, N, dw_g, dw_fc, db_g, db_fc, stream, accumulate, 0);
}

cudaError_t launch_fused_w_partials(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                                    int64_t M, int64_t K, int64_t N, float* dw_part, float* db_part,
                                    const FwPlan& plan, cudaStream_t stream) {
  if (plan.splits < 2) return cudaErrorInvalidValue;  // one split would write bf16 dw directly
  return launch_fw_kernel(x, dy, g, fc, nullptr, nullptr, M, K, N, dw_part, db_part, plan, stream, false);
}

}  // namespace swg
