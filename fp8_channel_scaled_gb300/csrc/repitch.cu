// repitch.cu -- copy the E4M3 operands x [M, K] and w [N, K], whose rows
// are not 16-byte aligned (K % 16 != 0, or a base address that is not
// 16-byte aligned), into a workspace whose rows are Kp bytes long (a multiple
// of 16 >= K: the library takes round_up(K, 64)), with the Kp - K pad bytes
// set to zero.  The tile kernel then
// reads the copies through TMA, which needs 16-byte row pitches.
//
// This is the per-call zero-padding pass the pages' Blackwell submission runs
// on live data ("Kimi K3 (256k)" page, sm_100 tcgen05 paragraph: K = 4127 is
// padded to 4128 by a padding kernel on every forward, never cached), here
// padding only to the next multiple of 64 bytes.  Zero bytes add exactly
// nothing to a dot product, so results equal the unpadded ones.
//
// One warp copies a segment of 64, 96 or 128 output chunks (the width that
// leaves the fewest lanes idle at the row's end: 96 for K = 4127) of one row
// of the stacked [x; w] matrix, issuing all its loads before using any, so
// that even a copy of a few thousand rows has tens of thousands of loads in
// flight at once.  Output chunk j of a row (bytes
// [16 j, 16 j + 16)) is bytes [sh, sh + 16) of the two aligned 16-byte source
// words at abase + 16 j and abase + 16 (j + 1), where abase is the row start
// rounded down to 16 bytes and sh the remainder: lane l loads the first word
// of its chunk, takes the second from lane l + 1 by shuffles (lane 31 loads
// it), shifts, masks bytes past K and stores 16 bytes.  Loads and stores are
// coalesced along the row.  No load touches a 16-byte word that holds no byte
// of the row.
#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"

namespace fp8g {
namespace {

constexpr int kThreads = 256;

// 16-byte read-only load with an L2 eviction policy: the source rows are read
// once, so they are marked evict-first and do not push the copies (read next
// by the GEMM) or other resident data out of L2 (K = 4127 call: 35.15 ->
// 34.62 us; keeping the copies with an evict-last store gained no more).
__device__ __forceinline__ uint4 ldg_nc_v4_policy(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
constexpr int kWarps = kThreads / 32;

// kU output chunks per lane, 32 kU per warp (one row segment).
template <int kU>
__global__ void __launch_bounds__(kThreads) repitch_kernel(const RepitchArgs a,
                                                           const int segs_per_row) {
  constexpr int kSegChunks = 32 * kU;
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t lane = threadIdx.x & 31u;
  const long long g = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const long long r = g / segs_per_row;
  if (r >= a.rows_x + a.rows_w) return;
  const int j0 = static_cast<int>(g - r * segs_per_row) * kSegChunks;
  const bool is_w = r >= a.rows_x;
  const long long rr = is_w ? r - a.rows_x : r;
  const uint8_t* src = (is_w ? a.w : a.x) + rr * (is_w ? a.ldw : a.ldx);
  uint8_t* dst = (is_w ? a.wo : a.xo) + rr * a.Kp;
  const uint32_t sh = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
  const uint8_t* abase = src - sh;
  const long long span = static_cast<long long>(sh) + a.K;  // bytes from abase to the row's end
  const int cpr = a.Kp / 16;                               // output chunks per row
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const uint64_t pol = l2_policy_evict_first();
  // every load of the segment is issued before any is used: the words of
  // the lanes' own chunks, and lane 31's word past each 32-chunk run
  uint4 lo[kU], tail[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const long long off = 16LL * (j0 + u * 32 + static_cast<int>(lane));
    lo[u] = off < span ? ldg_nc_v4_policy(abase + off, pol) : zero;
    tail[u] = zero;
    if (lane == 31u && sh != 0u && off + 16 < span)
      tail[u] = ldg_nc_v4_policy(abase + off + 16, pol);
  }
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int j = j0 + u * 32 + static_cast<int>(lane);
    uint4 hi;
    hi.x = __shfl_down_sync(0xffffffffu, lo[u].x, 1);
    hi.y = __shfl_down_sync(0xffffffffu, lo[u].y, 1);
    hi.z = __shfl_down_sync(0xffffffffu, lo[u].z, 1);
    hi.w = __shfl_down_sync(0xffffffffu, lo[u].w, 1);
    if (lane == 31u) hi = tail[u];
    if (j < cpr) {
      const uint4 v = keep_bytes(realign16(lo[u], hi, sh), a.K - 16 * j);
      *reinterpret_cast<uint4*>(dst + 16LL * j) = v;
    }
  }
}

}  // namespace

cudaError_t launch_repitch(const RepitchArgs& a, cudaStream_t s) {
  const long long rows = a.rows_x + a.rows_w;
  if (rows <= 0 || a.Kp <= 0) return cudaSuccess;
  // segment width: the fewest idle lane slots over a row (ties: wider)
  const int cpr = a.Kp / 16;
  int best_u = 2, best_slots = 0;
  for (int u = 2; u <= 4; ++u) {
    const int slots = (cpr + 32 * u - 1) / (32 * u) * (32 * u);
    if (best_slots == 0 || slots <= best_slots) {
      best_u = u;
      best_slots = slots;
    }
  }
  const int segs = (cpr + 32 * best_u - 1) / (32 * best_u);
  const long long blocks = (rows * segs + kWarps - 1) / kWarps;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  set_pdl(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  switch (best_u) {
    case 2: return cudaLaunchKernelEx(&cfg, repitch_kernel<2>, a, segs);
    case 3: return cudaLaunchKernelEx(&cfg, repitch_kernel<3>, a, segs);
    default: return cudaLaunchKernelEx(&cfg, repitch_kernel<4>, a, segs);
  }
}

}  // namespace fp8g
