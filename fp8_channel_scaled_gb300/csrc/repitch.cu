// repitch.cu -- copy the E4M3 operands x [M, K] and w [N, K], whose rows
// are not 16-byte aligned (K % 16 != 0, or a base address that is not
// 16-byte aligned), into a workspace whose rows are Kp = round_up(K, 16)
// bytes long, with the Kp - K pad bytes set to zero.  The tile kernel then
// reads the copies through TMA, which needs 16-byte row pitches.
//
// This is the per-call zero-padding pass the pages' Blackwell submission runs
// on live data ("Kimi K3 (256k)" page, sm_100 tcgen05 paragraph: K = 4127 is
// padded to 4128 by a padding kernel on every forward, never cached), here
// padding only to the next multiple of 16 bytes.  Zero bytes add exactly
// nothing to a dot product, so results equal the unpadded ones.
//
// One thread produces one aligned 16-byte output chunk from the (at most)
// two aligned 16-byte source words that hold it, so loads and stores are
// both 16 bytes wide and coalesced along the row; each thread keeps four
// chunks in flight.  No load touches a 16-byte word that holds no byte of
// the operand.
#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"

namespace fp8g {
namespace {

constexpr int kThreads = 256;
constexpr int kIlp = 4;

__device__ __forceinline__ void chunk_of(const RepitchArgs& a, long long u, const uint8_t*& src,
                                         uint8_t*& dst, int& valid) {
  const long long cpr = a.Kp / 16;
  const bool is_w = u >= a.chunks_x;
  const long long v = is_w ? u - a.chunks_x : u;
  const long long r = v / cpr;
  const int c = static_cast<int>(v - r * cpr);
  const int kc = 16 * c;
  src = (is_w ? a.w : a.x) + r * a.K + kc;
  dst = (is_w ? a.wo : a.xo) + r * a.Kp + kc;
  valid = min(16, a.K - kc);
}

__global__ void __launch_bounds__(kThreads) repitch_kernel(const RepitchArgs a) {
  const long long total = a.chunks_x + a.chunks_w;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long base = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; base < total;
       base += stride * kIlp) {
    uint4 lo[kIlp], hi[kIlp];
    uint32_t sh[kIlp];
    int valid[kIlp];
    uint8_t* dst[kIlp];
#pragma unroll
    for (int i = 0; i < kIlp; ++i) {
      const long long u = base + i * stride;
      lo[i] = make_uint4(0, 0, 0, 0);
      hi[i] = make_uint4(0, 0, 0, 0);
      sh[i] = 0;
      valid[i] = 0;
      dst[i] = nullptr;
      if (u < total) {
        const uint8_t* src;
        chunk_of(a, u, src, dst[i], valid[i]);
        sh[i] = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src) & 15u);
        const uint8_t* w0 = src - sh[i];
        lo[i] = ldg_nc_v4(w0);
        if (sh[i] != 0u && valid[i] > 16 - static_cast<int>(sh[i])) hi[i] = ldg_nc_v4(w0 + 16);
      }
    }
#pragma unroll
    for (int i = 0; i < kIlp; ++i) {
      if (dst[i]) {
        const uint4 v = keep_bytes(realign16(lo[i], hi[i], sh[i]), valid[i]);
        *reinterpret_cast<uint4*>(dst[i]) = v;
      }
    }
  }
}

}  // namespace

cudaError_t launch_repitch(const RepitchArgs& a, int sm_count, cudaStream_t s) {
  const long long total = a.chunks_x + a.chunks_w;
  if (total <= 0) return cudaSuccess;
  long long blocks = (total + static_cast<long long>(kThreads) * kIlp - 1) /
                     (static_cast<long long>(kThreads) * kIlp);
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  repitch_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace fp8g
