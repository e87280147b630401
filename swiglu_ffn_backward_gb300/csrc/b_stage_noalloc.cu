// swiglu_bwd_b_noalloc: the b stage for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc and cannot keep a workspace buffer
// between calls: for example a host framework whose memory pool owns all of
// device memory and forbids side allocations, or a latency-critical loop that
// cannot afford cudaMalloc's implicit device synchronisation. The regular
// swiglu_bwd_b needs a caller-provided workspace for its fp32 column partials;
// this entry point instead keeps them in a fixed array compiled into the
// library (kScratchBytes, 4 MiB), which every GPU that loads the library holds
// until the process exits. It allocates nothing and calls no allocating
// routine.
//
// The array is shared by every call on a device and keeps the last call's
// contents. Nothing in it needs to start at zero: each call writes every
// partial it later reads. Calls that overlap on the GPU (for example on two
// streams at once) race on the array and give wrong column sums; serialise
// them.
//
// Host code must not pass the array's name to a kernel: on the host it is a
// stand-in, not a device address. Every call looks the device address up with
// cudaGetSymbolAddress on the current device (the device the call launches
// on), so the address is never stale, not even after a cudaDeviceReset. The
// first call on a device also loads the library's device code there; make
// that first call before any stream capture.
#include <cuda_runtime.h>

#include "../../include/swiglu_bwd.h"
#include "swg_launch.h"

namespace {

constexpr size_t kScratchBytes = SWG_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_b_scratch[kScratchBytes];

// device address of g_b_scratch on the current device, looked up on every call
swg_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_b_scratch) != cudaSuccess || p == nullptr) return SWG_ERR_CUDA;
  *out = p;
  return SWG_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

}  // namespace

extern "C" swg_status swiglu_bwd_b_noalloc(const void* dy, const void* g, const void* fc, void* dg, void* dfc,
                                           void* db_g, void* db_fc, int64_t M, int64_t N,
                                           swg_stream_t stream) {
  if (M < 0 || N < 0) return SWG_ERR_PARAM_INVALID;
  if (M > 0x7fffffffLL || N > 0x7fffffffLL || (N % 8) != 0) return SWG_ERR_UNSUPPORTED;
  if (N == 0) return SWG_OK;
  if (!db_g || !db_fc || (M > 0 && (!dy || !g || !fc || !dg || !dfc))) return SWG_ERR_NULLPTR;
  const void* all[] = {dy, g, fc, dg, dfc, db_g, db_fc};
  for (const void* p : all)
    if (!aligned16(p)) return SWG_ERR_UNSUPPORTED;
  const int64_t mn = M * N * 2;
  const void* outs[] = {dg, dfc, db_g, db_fc};
  const int64_t osz[] = {mn, mn, N * 2, N * 2};
  const void* ins[] = {dy, g, fc};
  for (int i = 0; i < 4; ++i) {
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], osz[i], outs[j], osz[j])) return SWG_ERR_PARAM_INVALID;
    for (int j = 0; j < 3; ++j)
      if (overlaps(outs[i], osz[i], ins[j], mn)) return SWG_ERR_PARAM_INVALID;
  }
  // the column partials must fit the built-in array (always true for N <= 524288)
  if (swg::b_workspace_bytes(M, N) > kScratchBytes) return SWG_ERR_WORKSPACE;

  int dev = 0, maj = 0, min = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SWG_ERR_CUDA;
  if (maj != 10 || min != 3) return SWG_ERR_UNSUPPORTED;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    if (cudaMemsetAsync(db_g, 0, static_cast<size_t>(N) * 2, s) != cudaSuccess ||
        cudaMemsetAsync(db_fc, 0, static_cast<size_t>(N) * 2, s) != cudaSuccess)
      return SWG_ERR_CUDA;
    return SWG_OK;
  }
  void* scratch = nullptr;
  const swg_status st = scratch_address(&scratch);
  if (st != SWG_OK) return st;
  const cudaError_t e = swg::launch_b_stage(
      static_cast<const uint16_t*>(dy), static_cast<const uint16_t*>(g), static_cast<const uint16_t*>(fc),
      static_cast<uint16_t*>(dg), static_cast<uint16_t*>(dfc), static_cast<uint16_t*>(db_g),
      static_cast<uint16_t*>(db_fc), M, N, scratch, s);
  return e == cudaSuccess ? SWG_OK : SWG_ERR_CUDA;
}
