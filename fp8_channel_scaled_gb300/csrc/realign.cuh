// realign.cuh -- operand loader for rows that are not 16-byte aligned.
//
// A TMA tensor map needs every row pitch to be a multiple of 16 bytes, so a
// row-major E4M3 matrix with K % 16 != 0 (e.g. K = 4127) cannot be tiled by
// TMA.  Instead of padding a copy on the host or in a separate pass (what
// the pages' submissions do for K = 4127: "Kimi K3 (256k)" page, SM100
// tcgen05 paragraph; "claude-fable-5" page, SM120 funnel-shift pad-copy
// paragraph), producer threads read each row segment with 16-byte aligned
// loads, shift the bytes into place in registers, zero everything at
// k >= K, and write the result straight into the 128-byte-swizzled K-major
// shared-memory layout the tensor cores read.  Zero bytes contribute exactly
// nothing to the dot product, so the result equals the unpadded one.
//
// Every global load touches a 16-byte word that contains at least one byte
// of the requested row segment, so no load leaves the operand's own
// 16-byte-aligned granules.
#pragma once

#include "ptx.cuh"

namespace fp8g {

// Bytes [sh, sh+16) of the 32-byte little-endian value hi:lo.
__device__ __forceinline__ uint4 realign16(const uint4& lo, const uint4& hi, uint32_t sh) {
  const uint32_t u0 = lo.x, u1 = lo.y, u2 = lo.z, u3 = lo.w;
  const uint32_t u4 = hi.x, u5 = hi.y, u6 = hi.z, u7 = hi.w;
  const uint32_t q = sh >> 2;
  const uint32_t bits = (sh & 3u) * 8u;
  uint32_t t0, t1, t2, t3, t4;
  if (q == 0) {
    t0 = u0; t1 = u1; t2 = u2; t3 = u3; t4 = u4;
  } else if (q == 1) {
    t0 = u1; t1 = u2; t2 = u3; t3 = u4; t4 = u5;
  } else if (q == 2) {
    t0 = u2; t1 = u3; t2 = u4; t3 = u5; t4 = u6;
  } else {
    t0 = u3; t1 = u4; t2 = u5; t3 = u6; t4 = u7;
  }
  uint4 r;
  r.x = __funnelshift_r(t0, t1, bits);
  r.y = __funnelshift_r(t1, t2, bits);
  r.z = __funnelshift_r(t2, t3, bits);
  r.w = __funnelshift_r(t3, t4, bits);
  return r;
}

// Keep the first `valid` bytes (0..16) of v, zero the rest.
__device__ __forceinline__ uint4 keep_bytes(uint4 v, int valid) {
  auto m = [](int nb) -> uint32_t {
    return nb >= 4 ? 0xFFFFFFFFu : (nb <= 0 ? 0u : ((1u << (8 * nb)) - 1u));
  };
  v.x &= m(valid);
  v.y &= m(valid - 4);
  v.z &= m(valid - 8);
  v.w &= m(valid - 12);
  return v;
}

// Copy rows [r0, r0+R) x bytes [k0, k0+128) of a row-major byte matrix with
// `rows_total` rows and pitch K bytes into the K-major 128-byte-swizzled
// shared-memory layout of one operand stage (row r, 16-byte chunk c at
// r * 128 + ((c ^ (r & 7)) << 4)), zero past rows_total and past K.  It is
// split into a load half and a store half, so that a producer issues all
// of a block's loads (even before it waits for the stage to be free) and
// then stores them: one memory latency per block, not one per batch of
// chunks.  The loads sit in registers, so a producer cannot keep enough in
// flight to stream at HBM rate; callers repitch instead when they can.
//
// Thread tid holds chunks u = i * NT + tid (i < PER): row u / 8, 16-byte
// chunk u % 8.  Since NT is a multiple of 8, lanes 8j .. 8j + 7 of a warp
// hold one row's 8 chunks in order, so the second source word of a chunk is
// the next lane's first word (taken by shuffle) except for a row's last
// chunk, which loads it.  A lane loads a word only if it holds a byte of the
// row: word start < row + K.
template <int R, int NT>
struct RealignRegs {
  static constexpr int PER = R * 8 / NT;
  static_assert((R * 8) % NT == 0 && NT % 32 == 0, "units must split evenly over warps");
  uint4 lo[PER];
  uint4 tail[PER];   // a row's last chunk: the word after it
  uint32_t sh[PER];
  int valid[PER];    // bytes of the chunk that are < K (<= 0: none)
};

template <int R, int NT>
__device__ __forceinline__ void realign_load(RealignRegs<R, NT>& g, const uint8_t* __restrict__ src,
                                             int rows_total, int K, int r0, int k0, int tid) {
#pragma unroll
  for (int i = 0; i < RealignRegs<R, NT>::PER; ++i) {
    const int u = i * NT + tid;
    const int r = u >> 3, c = u & 7;
    const int grow = r0 + r, kc = k0 + 16 * c;
    g.lo[i] = make_uint4(0, 0, 0, 0);
    g.tail[i] = make_uint4(0, 0, 0, 0);
    g.sh[i] = 0;
    g.valid[i] = 0;
    if (grow < rows_total) {
      const uint8_t* row = src + static_cast<size_t>(grow) * static_cast<size_t>(K);
      const uint32_t sh = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row + kc) & 15u);
      const uint8_t* base = row + kc - sh;  // aligned word holding byte kc
      g.sh[i] = sh;
      g.valid[i] = K - kc;
      // word [base, base + 16) holds row bytes iff base < row + K
      if (kc - static_cast<int>(sh) < K) g.lo[i] = ldg_nc_v4(base);
      if (c == 7 && sh != 0u && kc + 16 - static_cast<int>(sh) < K) g.tail[i] = ldg_nc_v4(base + 16);
    }
  }
}

template <int R, int NT>
__device__ __forceinline__ void realign_store(uint32_t dst, const RealignRegs<R, NT>& g, int tid) {
#pragma unroll
  for (int i = 0; i < RealignRegs<R, NT>::PER; ++i) {
    const int u = i * NT + tid;
    const int r = u >> 3, c = u & 7;
    uint4 hi;
    hi.x = __shfl_down_sync(0xffffffffu, g.lo[i].x, 1);
    hi.y = __shfl_down_sync(0xffffffffu, g.lo[i].y, 1);
    hi.z = __shfl_down_sync(0xffffffffu, g.lo[i].z, 1);
    hi.w = __shfl_down_sync(0xffffffffu, g.lo[i].w, 1);
    if (c == 7) hi = g.tail[i];
    const uint4 v = keep_bytes(realign16(g.lo[i], hi, g.sh[i]), g.valid[i]);
    sts_v4(dst + static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)), v);
  }
}

}  // namespace fp8g
