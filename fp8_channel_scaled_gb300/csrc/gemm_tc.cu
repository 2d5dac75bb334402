// gemm_tc.cu -- persistent, warp-specialised tcgen05 kernel for the scaled
// FP8 linear layer  y = bf16((x_e4m3 . w_e4m3^T, fp32 accumulate) * scale[n]).
//
// The design follows what the pages describe for the Blackwell tcgen05
// submission ("Kimi K3 (256k)" page, sm_100 tcgen05 paragraph: TMA loader
// warp + MMA warp + 4-warp epilogue, kind::f8f6f4 with fp32 accumulation in
// tensor memory, per-channel scale in the epilogue, bf16 out) and the SM90
// paragraph of the same page (persistent grid, multi-stage mbarrier ring,
// grouped rasterisation for L2 reuse), rebuilt for sm_103a:
//
//   warps 0-3  epilogue: tcgen05.ld of the fp32 accumulator (warp w owns
//              TMEM lanes 32w..32w+31 = tile rows), * scale[n], cvt.rn to
//              bf16, 16-byte global stores
//   warp  4    TMEM allocator + single-thread tcgen05.mma issuer
//   warps 5-6  TMA producers, one thread each (warp 5: x tiles, warp 6: w
//              tiles; one issuing thread alone cannot keep enough copies in
//              flight) -- or, with `realign`, warps 5-8 load rows whose pitch
//              is not a multiple of 16 bytes and write them into the
//              swizzled layout themselves
//
// Tile 128 x BN x 128 bytes of K per stage; the accumulator is double
// buffered in TMEM (2 x BN fp32 columns), so the epilogue of one tile runs
// under the mainloop of the next.  Tiles beyond M/N and K blocks beyond K are
// zero-filled by the TMA (or by the realigning loader); zero bytes add
// exactly nothing to the dot products.
//
// Every wait is bounded (see ptx.cuh): a wait that runs out records an error
// bit in the device error word and the CTA winds down, after waiting (again
// with a limit) for its own copies and MMAs in flight and freeing its TMEM.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"
#include "sched.cuh"

namespace fp8g {
namespace {

constexpr int kBM = 128;        // tile rows (M) = TMEM lanes
constexpr int kBK = 128;        // bytes (= E4M3 elements) of K per stage
constexpr int kMmaK = 32;       // K per tcgen05.mma kind::f8f6f4
constexpr int kEpiWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProdWarp0 = 5;

template <int BN, int STAGES, bool REALIGN>
struct Cfg {
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kProdWarps = REALIGN ? 4 : 2;
  static constexpr int kThreads = 32 * (kProdWarp0 + kProdWarps);
  static constexpr int kTmemCols = (2 * BN <= 256) ? 256 : 512;
  static constexpr int kBarOff = STAGES * kStageBytes;
  // full[S], empty[S], tfull[2], tempty[2], mma_done, then tmem holder + abort flag
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8 + 16;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(2 * BN <= kTmemCols, "two accumulators must fit in TMEM");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int BN, int STAGES, bool REALIGN>
__global__ void __launch_bounds__(Cfg<BN, STAGES, REALIGN>::kThreads, 1)
    fp8_linear_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const GemmArgs p,
                         const int num_m_blk, const int num_n_blk, const int group_m) {
  using C = Cfg<BN, STAGES, REALIGN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw_addr);

  const uint32_t bar0 = sbase + C::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 4);
  const uint32_t holder_addr = bar0 + 8u * C::kNumBars;
  volatile uint32_t* holder = reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOff + 8 * C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 8 * C::kNumBars + 4);
  auto sA = [&](int s) { return sbase + static_cast<uint32_t>(s * C::kStageBytes); };
  auto sB = [&](int s) { return sbase + static_cast<uint32_t>(s * C::kStageBytes + C::kABytes); };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), REALIGN ? 32u * C::kProdWarps : 2u);
      mbar_init(empty_bar(s), 1u);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1u);
      mbar_init(tempty_bar(a), static_cast<uint32_t>(kEpiWarps));
    }
    mbar_init(mma_done_bar, 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Global memory (operands, scales, y) is touched only after the preceding
  // grids of the stream have completed; the set-up above overlaps their tail.
  // Tensor memory is allocated only after the wait, so this CTA never holds
  // it while it waits for another grid.
  griddep_wait();
  if (warp == kMmaWarp) {
    tmem_alloc(holder_addr, C::kTmemCols);
    tmem_relinquish();
  }
  if (!REALIGN && warp == kProdWarp0 && lane == 0) tma_prefetch_desc(&tmA);
  if (!REALIGN && warp == kProdWarp0 + 1 && lane == 0) tma_prefetch_desc(&tmB);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *holder;
  // Our dependents may launch once every CTA of this grid holds its tensor
  // memory: a dependent CTA sharing an SM can then only wait for ours to
  // free it, never take it first.
  griddep_launch_dependents();

  const WaitCtx wc{p.err, abort_flag, p.budget_ns};
  const int num_tiles = num_m_blk * num_n_blk;
  const int num_kb = p.num_kb;

  if (warp >= kProdWarp0) {
    // ------------------------------------------------------------ producer
    if (!REALIGN) {
      if (lane == 0) {
        const bool is_a = warp == kProdWarp0;
        const CUtensorMap* map = is_a ? &tmA : &tmB;
        const uint32_t bytes = is_a ? C::kABytes : C::kBBytes;
        const uint32_t off = is_a ? 0u : static_cast<uint32_t>(C::kABytes);
        uint32_t stage = 0, phase = 0, issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
          int mb, nb;
          tile_coords(t, num_m_blk, num_n_blk, group_m, mb, nb);
          const int row = is_a ? mb * kBM : nb * BN;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, wc, kErrWaitProducer)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(stage), bytes);
            tma_load_2d(sbase + static_cast<uint32_t>(stage * C::kStageBytes) + off, map,
                        full_bar(stage), kb * kBK, row);
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // Every load issued must have landed before the CTA may exit.  In a
        // normal run the MMA warp already waited for all of them.
        for (int s = 0; s < STAGES; ++s) {
          if (issued > static_cast<uint32_t>(s)) {
            const uint32_t n_s = (issued - 1u - s) / STAGES + 1u;
            drain_wait(full_bar(s), (n_s - 1u) & 1u, p.err, p.budget_ns);
          }
        }
      }
      __syncwarp();
    } else {
      const int ptid = static_cast<int>(threadIdx.x) - kProdWarp0 * 32;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, num_m_blk, num_n_blk, group_m, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb) {
          // x rows in one load round (issued before waiting for the stage),
          // then w rows in two rounds of BN / 2 rows
          RealignRegs<kBM, 128> ga;
          realign_load(ga, p.x, p.M, p.K, mb * kBM, kb * kBK, ptid);
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, wc, kErrWaitProducer)) {
            ok = false;
            break;
          }
          realign_store(sA(stage), ga, ptid);
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            RealignRegs<BN / 2, 128> gb;
            realign_load(gb, p.w, p.N, p.K, nb * BN + h * (BN / 2), kb * kBK, ptid);
            realign_store(sB(stage) + static_cast<uint32_t>(h * (BN / 2) * 128), gb, ptid);
          }
          fence_proxy_async_smem();
          mbar_arrive(full_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, wc, kErrWaitMma)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, wc, kErrWaitMma)) {
            ok = false;
            break;
          }
          // TMA data reach the MMA through the full barrier alone; operands written
          // by producer threads (generic proxy) additionally need the tcgen05 fence
          if (REALIGN) tc_fence_after_sync();
          const uint64_t a_desc = sdesc_kmajor_sw128(sA(stage));
          const uint64_t b_desc = sdesc_kmajor_sw128(sB(stage));
#pragma unroll
          for (int k = 0; k < kBK / kMmaK; ++k) {
            // +32 bytes along K inside the swizzled 128-byte row = +2 in the
            // descriptor's address field (16-byte units)
            tc_mma_f8(d_tmem, a_desc + 2u * k, b_desc + 2u * k, kIdesc,
                      (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all MMAs issued by this thread must be complete before teardown
      tc_commit(mma_done_bar);
      drain_wait(mma_done_bar, 0u, p.err, p.budget_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    uint32_t acc = 0, acc_phase = 0;
    const bool zero_acc = (num_kb == 0);
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, num_m_blk, num_n_blk, group_m, mb, nb);
      if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, wc, kErrWaitEpilogue)) break;
      tc_fence_after_sync();
      const int row = mb * kBM + static_cast<int>(warp) * 32 + static_cast<int>(lane);
      const uint32_t t_row = tmem_base + ((warp * 32u) << 16) + acc * BN;
      uint16_t* yrow = p.y + static_cast<size_t>(row) * static_cast<size_t>(p.N);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + c * 32, v);
        tmem_ld_wait();
        const int col0 = nb * BN + c * 32;
        const float sc = (col0 + static_cast<int>(lane) < p.N) ? __ldg(p.scale + col0 + lane) : 0.f;
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float s0 = __shfl_sync(0xffffffffu, sc, 2 * j);
          const float s1 = __shfl_sync(0xffffffffu, sc, 2 * j + 1);
          const float a0 = zero_acc ? 0.f : __uint_as_float(v[2 * j]);
          const float a1 = zero_acc ? 0.f : __uint_as_float(v[2 * j + 1]);
          packed[j] = pack_bf16x2(a0 * s0, a1 * s1);
        }
        if (row < p.M) {
          if (p.vec_store && col0 + 32 <= p.N) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                  packed[4 * q + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (col0 + j < p.N)
                yrow[col0 + j] = static_cast<uint16_t>((j & 1) ? (packed[j >> 1] >> 16)
                                                               : (packed[j >> 1] & 0xFFFFu));
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ------------------------------------------------------------------ dispatch
using KernelFn = void (*)(CUtensorMap, CUtensorMap, GemmArgs, int, int, int);

struct Entry {
  int bn, stages;
  bool realign;
  const void* fn;
  int smem, threads;
};

template <int BN, int S, bool R>
Entry make_entry() {
  return Entry{BN, S, R, reinterpret_cast<const void*>(&fp8_linear_tc_kernel<BN, S, R>),
               Cfg<BN, S, R>::kSmemBytes, Cfg<BN, S, R>::kThreads};
}

// N tiles and pipeline depths that are built: for each N tile the deepest
// ring that fits in shared memory (and one shallower ring), plus the
// realigning-producer variants used when no workspace can be had.  64-wide
// tiles serve 129-256 rows with few N blocks: twice the CTAs of 128-wide
// tiles stream the weight (256 x 4096 x 4096: 13.3 us against 14.2 us).
const Entry kEntries[] = {
    make_entry<256, 4, false>(), make_entry<256, 3, false>(), make_entry<224, 5, false>(),
    make_entry<224, 4, false>(), make_entry<192, 5, false>(), make_entry<160, 6, false>(),
    make_entry<128, 7, false>(), make_entry<128, 6, false>(), make_entry<64, 9, false>(),
    make_entry<64, 8, false>(),  make_entry<256, 4, true>(),  make_entry<224, 4, true>(),
    make_entry<128, 6, true>(),
};

const Entry* find(int bn, int stages, bool realign) {
  for (const Entry& e : kEntries)
    if (e.bn == bn && e.stages == stages && e.realign == realign) return &e;
  return nullptr;
}

}  // namespace

bool tc_config_supported(int bn, int stages, bool realign) {
  return find(bn, stages, realign) != nullptr;
}

int tc_smem_bytes(int bn, int stages, bool realign) {
  const Entry* e = find(bn, stages, realign);
  return e ? e->smem : -1;
}

int tc_threads(bool realign) { return 32 * (kProdWarp0 + (realign ? 4 : 2)); }

int tc_max_stages(int bn, bool realign, int smem_optin) {
  int best = 0;
  for (const Entry& e : kEntries)
    if (e.bn == bn && e.realign == realign && e.smem <= smem_optin && e.stages > best)
      best = e.stages;
  return best;
}

cudaError_t tc_blocks_per_sm(int bn, int stages, bool realign, int* out) {
  const Entry* e = find(bn, stages, realign);
  if (!e) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, e->fn, e->threads,
                                                       static_cast<size_t>(e->smem));
}

cudaError_t tc_prepare(int bn, int stages, bool realign) {
  const Entry* e = find(bn, stages, realign);
  if (!e) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(e->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, e->smem);
}

cudaError_t launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                      const TcConfig& c, cudaStream_t s) {
  const Entry* e = find(c.bn, c.stages, c.realign);
  if (!e) return cudaErrorInvalidValue;
  const int num_m_blk = (a.M + kBM - 1) / kBM;
  const int num_n_blk = (a.N + c.bn - 1) / c.bn;
  CUtensorMap mA = tmA, mB = tmB;
  GemmArgs args = a;
  int gm = c.group_m;
  void* params[] = {&mA, &mB, &args, const_cast<int*>(&num_m_blk), const_cast<int*>(&num_n_blk),
                    &gm};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(e->threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(e->smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  set_pdl(attr[0]);
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, e->fn, params);
}

}  // namespace fp8g
