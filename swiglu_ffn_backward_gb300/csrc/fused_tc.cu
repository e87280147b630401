// Fused variant of the SwiGLU-FFN backward: the b-stage math runs inside the
// GEMMs' operand producer, so dg and dfc are formed tile by tile in shared
// memory and never written to (or read back from) HBM.
//
// Sources: "PyPTO-Gym in practice: the fused SwiGLU backward operator",
// "Algorithm overview and formulas" items 1-4 (the math of every stage); the
// recompute-instead-of-store principle stated in the Ascend C backward blog
// post (Swish section: recompute sigma in the backward rather than keep it).
//
// Two kernels, both one CTA per SM with eleven warps:
//   warp 0 lane 0   TMA producer of the raw ring (dy, g, fc tiles)
//   warp 10 lane 0  TMA producer of the operand ring (W chunks, or x chunks)
//   warp 1          TMEM allocation (512 columns); lane 0 issues tcgen05.mma
//   warps 2-9       transform: read dy, g, fc from shared memory, compute dg,
//                   dfc in fp32, write them as bf16 IN PLACE over g and fc
//                   (the TMA swizzle permutes 16-byte chunks within each row
//                   the same way for all three tiles, so an element-wise map
//                   needs no layout work); then the epilogue, two warps per
//                   32-lane TMEM quarter, one per 256-column accumulator half.
//
// fused x (FX): D = dx[m0:m0+128, k0:k0+512] in two 256-column accumulators.
//   Stages of 64 reduction columns, 128-byte swizzle: a raw stage is 3 x 16 KB,
//   an operand entry is one W chunk [256 k x 64 n] (32 KB). A = dg or dfc
//   [128 m x 64 n] (K-major, in the g/fc slots), B = W_g / W_fc. Each dg
//   element is computed once per 512 columns of dx (once when K <= 512); dg,
//   dfc can also be written to HBM as optional outputs.
// fused w (FW): D = [dw_g^T ; dw_fc^T][n0:n0+64, k0:k0+512]: the A operand
//   stacks 64 columns of dg over the same 64 columns of dfc (MN-major, 128-byte
//   swizzle; the g slot and the fc slot are the two 64-element MN chunks,
//   LBO = 8 KB apart), so one accumulator pair holds both outputs for all k.
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

constexpr int kThreads = 352;
constexpr int kXThreads = 256;  // transform / epilogue threads (warps 2-9)
constexpr int kRingWarp = 10;
constexpr int kClusterX = 4;  // CTAs sharing each W chunk in the fused x kernel
constexpr int kClusterW = 4;  // CTAs sharing each x chunk in the fused w kernel
constexpr uint32_t kTmemCols = 512;

template <int MODE>
struct Cfg;
template <>
struct Cfg<kFX> {
  static constexpr int kRawRows = 128;     // m rows of a raw tile
  static constexpr int kRowBytes = 128;    // 64 bf16 reduction columns, 128-byte swizzle
  static constexpr int kRawStages = 2;
  static constexpr int kEntryBytes = 32768;
  static constexpr int kEntries = 4;
};
template <>
struct Cfg<kFW> {
  static constexpr int kRawRows = 64;
  static constexpr int kRowBytes = 128;    // 64 bf16 columns of n, 128-byte swizzle
  static constexpr int kRawStages = 4;
  static constexpr int kEntryBytes = 32768;
  static constexpr int kEntries = 4;
};

template <int MODE>
struct __align__(1024) FSmem {
  using C = Cfg<MODE>;
  static constexpr int kSlot = C::kRawRows * C::kRowBytes;
  uint8_t ring[C::kEntries][C::kEntryBytes];
  uint8_t raw[C::kRawStages][3][kSlot];  // dy, g (-> dg), fc (-> dfc)
  uint64_t raw_full[C::kRawStages];
  uint64_t raw_empty[C::kRawStages];
  uint64_t a_ready[C::kRawStages];
  uint64_t ring_full[C::kEntries];
  uint64_t ring_empty[C::kEntries];
  uint64_t accum;
  uint32_t tmem_base;
  volatile uint32_t abort_flag;
  volatile uint32_t raw_issued, raw_consumed, ring_issued, ring_consumed;
};

struct FusedArgs {
  int M, K, N;
  uint32_t* status;
  int tiles_k;  // 512-column blocks of K
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
  int x3d;  // x entries come from one 3-D box (else four 2-D boxes)
};

template <int MODE>
__device__ __forceinline__ void flag_timeout(FSmem<MODE>& s, uint32_t* status) {
  if (status != nullptr) atomicOr(status, kStatusTimeout);
  s.abort_flag = 1u;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
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
    float g0, f0, g1, f1;
    swiglu_grad_elem(bf16lo(dyw[i]), bf16lo(gw[i]), bf16lo(fw[i]), g0, f0);
    swiglu_grad_elem(bf16hi(dyw[i]), bf16hi(gw[i]), bf16hi(fw[i]), g1, f1);
    sg[2 * i] += g0;
    sg[2 * i + 1] += g1;
    sf[2 * i] += f0;
    sf[2 * i + 1] += f1;
    og[i] = pack_bf16x2(g0, g1);
    of[i] = pack_bf16x2(f0, f1);
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
                 const __grid_constant__ CUtensorMap tm_b1, const FusedArgs args) {
  using S = FSmem<MODE>;
  using C = Cfg<MODE>;
  constexpr int kRS = C::kRawStages;
  constexpr int kRE = C::kEntries;
  constexpr int kRows = C::kRawRows;
  constexpr int kSlot = S::kSlot;
  extern __shared__ uint8_t smem_raw[];
  S& s = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- tile coordinates
  const uint32_t crank = CS > 1 ? cluster_ctarank() : 0u;
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << CS) - 1u);
  int m0 = 0, n0 = 0, k0 = 0, kt = 0, split = 0, nst = 0, kb_begin = 0;
  if (MODE == kFX) {
    // clusters of CS consecutive m tiles share kt (and so every W chunk)
    const int cid = blockIdx.x / CS;
    kt = cid % args.tiles_k;
    m0 = ((cid / args.tiles_k) * CS + static_cast<int>(crank)) * 128;
    k0 = kt * 512;
    nst = (args.N + 63) / 64;  // raw stages: 64 columns of n each
  } else {
    int t = blockIdx.x;
    const int nt = t % args.tiles_n;
    t /= args.tiles_n;
    kt = t % args.tiles_k;
    split = t / args.tiles_k;
    n0 = nt * 64;
    k0 = kt * 512;
    kb_begin = split * args.kb_per;
    nst = min(args.nkb_total, kb_begin + args.kb_per) - kb_begin;  // raw stages: 64 rows of m each
  }
  const int nh = (args.K - k0) > 256 ? 2 : 1;  // 256-column accumulator halves in use
  const int entries_per_stage = (MODE == kFX) ? 2 * nh : nh;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRS; ++i) {
      mbar_init(&s.raw_full[i], 1);
      mbar_init(&s.raw_empty[i], 1);
      mbar_init(&s.a_ready[i], kXThreads);
    }
    for (int i = 0; i < kRE; ++i) {
      mbar_init(&s.ring_full[i], 1);
      mbar_init(&s.ring_empty[i], CS);  // released by all CTAs of the cluster
    }
    mbar_init(&s.accum, 1);
    s.abort_flag = 0u;
    s.raw_issued = s.raw_consumed = s.ring_issued = s.ring_consumed = 0u;
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
    // ------------------------------------------------------------ raw producer
    if (lane == 0) {
      for (int i = 0; i < nst && !s.abort_flag; ++i) {
        const int r = i % kRS;
        if (i >= kRS && !mbar_wait(&s.raw_empty[r], ((i / kRS) - 1) & 1)) {
          flag_timeout(s, args.status);
          break;
        }
        const int c0 = MODE == kFX ? i * 64 : n0;               // n
        const int c1 = MODE == kFX ? m0 : (kb_begin + i) * 64;  // m
        mbar_arrive_expect_tx(&s.raw_full[r], 3 * kSlot);
        tma_load_2d(s.raw[r][0], &tm_dy, &s.raw_full[r], c0, c1);
        tma_load_2d(s.raw[r][1], &tm_g, &s.raw_full[r], c0, c1);
        tma_load_2d(s.raw[r][2], &tm_fc, &s.raw_full[r], c0, c1);
        s.raw_issued = i + 1;
      }
    }
  } else if (warp == kRingWarp) {
    // ------------------------------------------------------------ operand producer
    if (lane == 0) {
      const int total = nst * entries_per_stage;
      for (int j = 0; j < total && !s.abort_flag; ++j) {
        const int e = j % kRE;
        if (j >= kRE && !mbar_wait(&s.ring_empty[e], ((j / kRE) - 1) & 1)) {
          flag_timeout(s, args.status);
          break;
        }
        const int i = j / entries_per_stage, q = j % entries_per_stage;
        mbar_arrive_expect_tx(&s.ring_full[e], C::kEntryBytes);  // all CS slices land here
        if (MODE == kFX) {
          const int p = q / nh, h = q % nh;  // W_g / W_fc, k half
          constexpr int kSliceRows = 256 / CS;
          uint8_t* dst = s.ring[e] + crank * kSliceRows * 128;
          const int kr = k0 + 256 * h + static_cast<int>(crank) * kSliceRows;
          if (CS > 1)
            tma_load_2d_mc(dst, p ? &tm_b1 : &tm_b0, &s.ring_full[e], i * 64, kr, kMask);
          else
            tma_load_2d(dst, p ? &tm_b1 : &tm_b0, &s.ring_full[e], i * 64, kr);
        } else {
          const int mrow = (kb_begin + i) * 64;
          const int kk = k0 + 256 * q;
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
        s.ring_issued = j + 1;
      }
      if (CS > 1 && !s.abort_flag) {
        // the peers' last releases arrive on this CTA's barriers: see them land
        // before this CTA can leave
        for (int j = max(0, total - kRE); j < total; ++j)
          if (!mbar_wait(&s.ring_empty[j % kRE], (j / kRE) & 1)) {
            flag_timeout(s, args.status);
            break;
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 256, MODE == kFW, MODE == kFW);
      uint32_t j = 0;
      bool ok = true;
      for (int i = 0; i < nst && ok; ++i) {
        const int r = i % kRS;
        if (!mbar_wait(&s.a_ready[r], (i / kRS) & 1)) {
          flag_timeout(s, args.status);
          break;
        }
        tc_fence_after();
        const uint32_t g_slot = smem_u32(s.raw[r][1]);
        for (int q = 0; q < entries_per_stage; ++q, ++j) {
          const int e = j % kRE;
          if (!mbar_wait(&s.ring_full[e], (j / kRE) & 1)) {
            flag_timeout(s, args.status);
            ok = false;
            break;
          }
          s.ring_consumed = j + 1;
          tc_fence_after();
          const uint32_t b_addr = smem_u32(s.ring[e]);
          if (MODE == kFX) {
            const int p = q / nh, h = q % nh;
            const uint32_t a_addr = g_slot + p * kSlot;  // dg or dfc
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(tmem + h * 256, smem_desc(a_addr + 32 * k, 16, 1024), smem_desc(b_addr + 32 * k, 16, 1024),
                        idesc, (i > 0 || p > 0 || k > 0) ? 1u : 0u);
          } else {
            const int h = q;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(tmem + h * 256, smem_desc(g_slot + 2048 * k, kSlot, 1024),
                        smem_desc(b_addr + 2048 * k, 8192, 1024), idesc, (i > 0 || k > 0) ? 1u : 0u);
          }
          if (CS > 1)
            umma_commit_mc(&s.ring_empty[e], kMask);  // release the entry in every CTA of the cluster
          else
            umma_commit(&s.ring_empty[e]);
        }
        umma_commit(&s.raw_empty[r]);
      }
      umma_commit(&s.accum);
    }
  } else {
    // ------------------------------------------------------------ transform
    const int t = threadIdx.x - 64;                // 0..255
    constexpr int kChunks = C::kRowBytes / 16;     // 16-byte chunks per row: 8
    constexpr int kGroups = kXThreads / kChunks;   // row groups: 32
    const int c = t % kChunks;                     // logical chunk (8 columns)
    const int rg = t / kChunks;
    const bool want_dg = (MODE == kFX) && kt == 0 && args.dg_out != nullptr;
    const bool want_db = (MODE == kFW) && kt == 0 && args.db_part != nullptr;
    float cg[8], cf[8];  // column sums (FW: over the CTA's whole M range)
#pragma unroll
    for (int e = 0; e < 8; ++e) cg[e] = cf[e] = 0.0f;
    // A thread whose wait runs out stops computing ("dead") but keeps taking
    // part in the arrivals (and, at the end, the named barriers).
    bool dead = false;
    for (int i = 0; i < nst; ++i) {
      const int r = i % kRS;
      if (!dead && !mbar_wait(&s.raw_full[r], (i / kRS) & 1)) {
        flag_timeout(s, args.status);
        dead = true;
      }
      if (s.abort_flag) dead = true;
      if (t == 0 && !dead) s.raw_consumed = i + 1;
      if (!dead) {
        const uint32_t sdy = smem_u32(s.raw[r][0]);
        const uint32_t sg = sdy + kSlot;
        const uint32_t sf = sdy + 2 * kSlot;
#pragma unroll
        for (int qq = 0; qq < kRows / kGroups; ++qq) {
          const int row = rg + kGroups * qq;
          // 128-byte swizzle: the 16-byte chunk index is XORed with row & 7
          const int phys = c ^ (row & 7);
          const uint32_t off = row * C::kRowBytes + (phys << 4);
          uint4 odg, odfc;
          grad8_sum(lds128(sdy + off), lds128(sg + off), lds128(sf + off), odg, odfc, cg, cf);
          sts128(sg + off, odg);
          sts128(sf + off, odfc);
          if (want_dg) {
            const int grow = m0 + row;
            const int gcol = i * 64 + c * 8;
            if (grow < args.M && gcol < args.N) {
              const int64_t o = static_cast<int64_t>(grow) * args.N + gcol;
              *reinterpret_cast<uint4*>(args.dg_out + o) = odg;
              *reinterpret_cast<uint4*>(args.dfc_out + o) = odfc;
            }
          }
        }
        fence_proxy_async_smem();  // dg, dfc written by this thread -> visible to the tensor core
      }
      mbar_arrive(&s.a_ready[r]);
    }

    const bool acc_ok = mbar_wait(&s.accum, 0);
    if (!acc_ok) flag_timeout(s, args.status);
    if (want_db) {
      // Column sums over the CTA's rows (rows beyond M are zero-filled by TMA
      // and add 0). Lanes l, l^8, l^16, l^24 share a chunk; the 8 warps are
      // combined through the first raw slot, idle once accum has fired (every
      // raw stage has been consumed by then).
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cg[e] += __shfl_xor_sync(0xffffffffu, cg[e], 8);
        cg[e] += __shfl_xor_sync(0xffffffffu, cg[e], 16);
        cf[e] += __shfl_xor_sync(0xffffffffu, cf[e], 8);
        cf[e] += __shfl_xor_sync(0xffffffffu, cf[e], 16);
      }
      named_sync_transform();
      float* scratch = reinterpret_cast<float*>(s.raw[0][0]);  // [8 warps][8 chunks][16]
      if (lane < 8) {
        float* p = scratch + ((warp - 2) * 8 + c) * 16;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = cg[e];
          p[8 + e] = cf[e];
        }
      }
      named_sync_transform();
      if (t < 128) {
        const int which = t >> 6;  // 0: dg, 1: dfc
        const int col = t & 63;
        const int gcol = n0 + col;
        if (!dead && acc_ok && gcol < args.N) {
          float v = 0.0f;
#pragma unroll
          for (int w = 0; w < 8; ++w) v += scratch[(w * 8 + (col >> 3)) * 16 + which * 8 + (col & 7)];
          args.db_part[static_cast<int64_t>(split) * 2 * args.N + which * args.N + gcol] = v;
        }
      }
    }

    // ------------------------------------------------------------ epilogue
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
        if (MODE == kFX) {
          const int row = m0 + r;
          if (row < args.M) {
            uint4* dst = reinterpret_cast<uint4*>(args.dx + static_cast<int64_t>(row) * args.K + kcol);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (kcol + 8 * j < args.K) dst[j] = pack8(v + 8 * j);
          }
        } else {
          const int prob = r >> 6;  // lanes 0-63: dw_g, 64-127: dw_fc
          const int n = n0 + (r & 63);
          if (n < args.N) {
            if (args.splits == 1) {
              uint16_t* dst = (prob ? args.dw_fc : args.dw_g) + n;
#pragma unroll 8
              for (int e = 0; e < 32; ++e) {
                const int k = kcol + e;
                if (k < args.K) {
                  const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[e]));
                  dst[static_cast<int64_t>(k) * args.N] = *reinterpret_cast<const uint16_t*>(&b);
                }
              }
            } else {
              float* dst = args.ws + static_cast<int64_t>(split * 2 + prob) * args.K * args.N + n;
#pragma unroll 8
              for (int e = 0; e < 32; ++e) {
                const int k = kcol + e;
                if (k < args.K) dst[static_cast<int64_t>(k) * args.N] = __uint_as_float(v[e]);
              }
            }
          }
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (threadIdx.x == 0 && s.abort_flag) {
    // drain: copies issued but never waited on must land before the CTA exits
    for (uint32_t i = s.raw_consumed; i < s.raw_issued; ++i)
      if (!mbar_wait(&s.raw_full[i % kRS], (i / kRS) & 1)) break;
    for (uint32_t i = s.ring_consumed; i < s.ring_issued; ++i)
      if (!mbar_wait(&s.ring_full[i % kRE], (i / kRE) & 1)) break;
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
                   const CUtensorMap& c, const CUtensorMap& d, const CUtensorMap& e, const FusedArgs& args) {
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
  return cudaLaunchKernelEx(&cfg, fused_kernel<MODE, CS>, a, b, c, d, e, args);
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
  CUtensorMap mdy, mg, mfc, mw0, mw1;
  const uint64_t rs = static_cast<uint64_t>(N) * 2;
  if (!encode_tmap_2d_bf16(&mdy, dy, N, M, rs, 64, 128) || !encode_tmap_2d_bf16(&mg, g, N, M, rs, 64, 128) ||
      !encode_tmap_2d_bf16(&mfc, fc, N, M, rs, 64, 128) ||
      !encode_tmap_2d_bf16(&mw0, w_g, N, K, rs, 64, 256 / CS) ||
      !encode_tmap_2d_bf16(&mw1, w_fc, N, K, rs, 64, 256 / CS))
    return cudaErrorInvalidValue;
  FusedArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.N = static_cast<int>(N);
  a.status = status_word_ptr();
  a.tiles_k = static_cast<int>((K + 511) / 512);
  a.dx = dx;
  a.dg_out = dg;
  a.dfc_out = dfc;
  const int64_t mclusters = ((M + 127) / 128 + CS - 1) / CS;  // tail CTAs run on zero-filled rows
  return launch<kFX, CS>(static_cast<unsigned>(mclusters * CS * a.tiles_k), stream, mdy, mg, mfc, mw0, mw1, a);
}

cudaError_t launch_fused_w(const uint16_t* x, const uint16_t* dy, const uint16_t* g, const uint16_t* fc,
                           uint16_t* dw_g, uint16_t* dw_fc, uint16_t* db_g, uint16_t* db_fc, int64_t M, int64_t K,
                           int64_t N, void* ws, const FwPlan& plan, cudaStream_t stream) {
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
  a.dw_g = dw_g;
  a.dw_fc = dw_fc;
  const size_t dw_part = plan.splits > 1 ? static_cast<size_t>(plan.splits) * 2 * K * N * sizeof(float) : 0;
  a.ws = static_cast<float*>(ws);
  a.db_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + al256(dw_part));
  a.splits = static_cast<int>(plan.splits);
  a.kb_per = static_cast<int>(plan.kb_per);
  a.nkb_total = static_cast<int>((M + 63) / 64);
  a.tiles_n = static_cast<int>(((N + 63) / 64 + CS - 1) / CS * CS);  // clusters of CS n tiles
  a.x3d = x3d;
  const int64_t ctas = plan.splits * a.tiles_k * a.tiles_n;
  cudaError_t e = launch<kFW, CS>(static_cast<unsigned>(ctas), stream, mdy, mg, mfc, mx3, mx2, a);
  if (e != cudaSuccess) return e;
  if (plan.splits > 1) {
    e = launch_w_split_reduce(static_cast<const float*>(ws), plan.splits, K, N, dw_g, dw_fc, stream);
    if (e != cudaSuccess) return e;
  }
  return launch_db_reduce(a.db_part, plan.splits, N, db_g, db_fc, stream);
}

}  // namespace swg
