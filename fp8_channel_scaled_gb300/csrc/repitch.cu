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
// chunks in flight.  A row holds at most 2^31 / 16 chunks (K < 2^31).  No load touches a 16-byte word that holds no byte of
// the operand.
#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"

namespace fp8g {
namespace {

constexpr int kThreads = 256;
constexpr int kIlp = 4;
constexpr int kRowsPerBlock = 8;

// Each block copies kRowsPerBlock consecutive rows of the stacked [x; w]
// matrix (M + N rows); its threads walk the rows' 16-byte output chunks with
// block-local 32-bit indices, kIlp chunks in flight per thread.
__global__ void __launch_bounds__(kThreads) repitch_kernel(const RepitchArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int cpr = a.Kp / 16;  // chunks per row
  const long long row0 = static_cast<long long>(blockIdx.x) * kRowsPerBlock;
  const long long rows_total = a.rows_x + a.rows_w;
  const long long left = rows_total - row0;
  const int rows_here = left < kRowsPerBlock ? static_cast<int>(left) : kRowsPerBlock;
  const int units = rows_here * cpr;
  for (int base = static_cast<int>(threadIdx.x); base < units; base += kThreads * kIlp) {
    uint4 lo[kIlp], hi[kIlp];
    uint32_t sh[kIlp];
    int valid[kIlp];
    uint8_t* dst[kIlp];
#pragma unroll
    for (int i = 0; i < kIlp; ++i) {
      const int u = base + i * kThreads;
      lo[i] = make_uint4(0, 0, 0, 0);
      hi[i] = make_uint4(0, 0, 0, 0);
      sh[i] = 0;
      valid[i] = 0;
      dst[i] = nullptr;
      if (u < units) {
        const int rl = u / cpr;
        const int kc = 16 * (u - rl * cpr);
        const long long r = row0 + rl;
        const bool is_w = r >= a.rows_x;
        const long long rr = is_w ? r - a.rows_x : r;
        const uint8_t* src = (is_w ? a.w : a.x) + rr * a.K + kc;
        dst[i] = (is_w ? a.wo : a.xo) + rr * a.Kp + kc;
        valid[i] = min(16, a.K - kc);
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

cudaError_t launch_repitch(const RepitchArgs& a, cudaStream_t s) {
  const long long rows = a.rows_x + a.rows_w;
  if (rows <= 0 || a.Kp <= 0) return cudaSuccess;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  set_pdl(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, repitch_kernel, a);
}

}  // namespace fp8g
