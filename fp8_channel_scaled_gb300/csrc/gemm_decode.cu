// gemm_decode.cu -- split-K tcgen05 kernel for skinny M (decode), for the
// scaled FP8 linear layer  y = bf16((x_e4m3 . w_e4m3^T, fp32 acc) * scale[n]).
//
// With M <= 64 the layer is a weight stream: every byte of w is used once
// and the arithmetic is small.  The pages' submissions use split-K with fp32
// partials for skinny M and reduce them in a second step ("Kimi K3 (256k)"
// page, SM90 and SM120 paragraphs: atomicAdd partials and a separate scaled
// finalize kernel; "claude-fable-5" page, Triton paragraph: fp32 partials
// plus a fused reduce/scale/cast kernel for M <= 64).  Here the whole thing
// is one launch and needs no global scratch:
//
//   * swap-AB: the MMA's A operand is a 128-row tile of w (n on TMEM lanes),
//     its B operand is all of x padded to MP rows (m on TMEM columns), so one
//     tcgen05.mma 128 x MP x 32 covers every token at once;
//   * each CTA of a thread-block cluster of `splits` CTAs owns one 128-row
//     n-tile and a contiguous range of 128-byte K blocks, streamed through a
//     TMA mbarrier ring (w with an L2 evict-first hint, x evict-last);
//   * the fp32 partial accumulators are parked in each CTA's shared memory
//     and summed across the cluster through distributed shared memory in a
//     fixed order (split 0, 1, ...), then scaled, rounded to bf16 and stored.
//
// Roles: warps 0-3 load (one thread issues TMA; all four with `realign`) and
// then act as the epilogue (warp w reads TMEM lanes 32w..32w+31); warp 4
// allocates TMEM and issues the MMAs.  All waits are bounded.
#include "kernels.h"
#include "ptx.cuh"
#include "realign.cuh"

namespace fp8g {
namespace {

constexpr int kBN = 128;   // rows of w per tile (MMA M, TMEM lanes)
constexpr int kBK = 128;   // bytes of K per stage
constexpr int kMmaK = 32;
constexpr int kMmaWarp = 4;
constexpr int kThreads = 160;
constexpr int kMaxSplits = 8;  // largest cluster the planner forms

template <int MP>
__host__ __device__ constexpr int tmem_cols_for() {
  return MP <= 32 ? 32 : (MP <= 64 ? 64 : (MP <= 128 ? 128 : 256));
}

// TMA-issuing warps of the decode producer: the largest divisor of the ring
// depth that is at most 4, so that every stage has exactly one owner.
template <int STAGES>
__host__ __device__ constexpr int issuers_for() {
  return STAGES % 4 == 0 ? 4 : (STAGES % 3 == 0 ? 3 : (STAGES % 2 == 0 ? 2 : 1));
}

// KBS: 128-byte K blocks per pipeline stage.  KBS > 1 loads the stage's w
// rows and x rows with one 3-D TMA box each (128 bytes x rows x KBS K
// blocks; the tensor maps step K blocks 128 bytes apart), which lands as KBS
// ordinary 128-byte-swizzled K-major tiles: one large copy per stage streams
// the weight with far fewer, larger transfers.
template <int MP, int STAGES, bool REALIGN, int KBS = 1>
struct DCfg {
  static constexpr int kABytes1 = kBN * kBK;  // one K block of w rows
  static constexpr int kBBytes1 = MP * kBK;   // one K block of x rows
  static constexpr int kABytes = kABytes1 * KBS;
  static constexpr int kBBytes = kBBytes1 * KBS;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kPartBytes = kBN * MP * 4;
  static constexpr int kDataBytes =
      STAGES * kStageBytes > kPartBytes ? STAGES * kStageBytes : kPartBytes;
  static constexpr int kBarOff = kDataBytes;
  // full[S], empty[S], acc_full, mma_done, then tmem holder + abort flag
  static constexpr int kNumBars = 2 * STAGES + 2;
  // the n-tile's 128 scales, staged for the reduction
  static constexpr int kScaleOff = (kBarOff + kNumBars * 8 + 16 + 15) / 16 * 16;
  static constexpr int kSmemBytes = 1024 + kScaleOff + kBN * 4;
  static constexpr int kTmemCols = tmem_cols_for<MP>();
  static_assert(MP % 32 == 0 && MP >= 32 && MP <= 256, "MP");
  static_assert(KBS == 1 || !REALIGN, "the realigning loader fills one K block per stage");
  static_assert(kABytes1 % 1024 == 0 && kBBytes1 % 1024 == 0, "K-block tiles on 1024-byte atoms");
};

template <int MP, int STAGES, bool REALIGN, int KBS = 1>
__global__ void __launch_bounds__(kThreads)
    fp8_linear_decode_kernel(const __grid_constant__ CUtensorMap tmW,
                             const __grid_constant__ CUtensorMap tmX, const GemmArgs p,
                             const int splits) {
  using C = DCfg<MP, STAGES, REALIGN, KBS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw_addr);

  const uint32_t bar0 = sbase + C::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t acc_full_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 1);
  const uint32_t holder_addr = bar0 + 8u * C::kNumBars;
  volatile uint32_t* holder =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOff + 8 * C::kNumBars);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(gbase + C::kBarOff + 8 * C::kNumBars + 4);
  auto sA = [&](int s) { return sbase + static_cast<uint32_t>(s * C::kStageBytes); };
  auto sB = [&](int s) { return sbase + static_cast<uint32_t>(s * C::kStageBytes + C::kABytes); };
  const uint32_t part = sbase;  // fp32 partials [MP][128], reuses the ring after the mainloop
  float* scale_s = reinterpret_cast<float*>(gbase + C::kScaleOff);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const int rank = static_cast<int>(cluster_ctarank());
  const int n_tile = static_cast<int>(blockIdx.x) / splits;
  const int n0 = n_tile * kBN;
  const int kb_begin = static_cast<int>((static_cast<long long>(p.num_kb) * rank) / splits);
  const int kb_end = static_cast<int>((static_cast<long long>(p.num_kb) * (rank + 1)) / splits);
  const int my_kb = kb_end - kb_begin;
  // pipeline stages of this CTA (the host makes my_kb a multiple of KBS)
  const int my_it = my_kb / KBS;
  // one split: the CTA owns whole outputs and stores them straight from
  // tensor memory (no parking, no cluster reduction)
  const bool direct = splits == 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), REALIGN ? 128u : 1u);
      mbar_init(empty_bar(s), 1u);
    }
    mbar_init(acc_full_bar, 1u);
    mbar_init(mma_done_bar, 1u);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // While the preceding grid of the stream drains, the TMA issuers ask L2 for
  // this CTA's first STAGES boxes of w: a prefetch delivers nothing to the
  // CTA, so the loads issued after the dependency wait below still observe
  // every write of the preceding grids, but the weight stream starts from L2
  // instead of paying the DRAM latency after the wait (decode 32 x 8192 x
  // 8192: 15.5 -> 14.6 us per call back to back; prefetching the first 16
  // boxes instead gained less, 14.9 us).
  if (!REALIGN && lane == 0 && static_cast<int>(warp) < issuers_for<STAGES>()) {
    tma_prefetch_desc(&tmW);
    const int pf = my_it < STAGES ? my_it : STAGES;
    for (int i = static_cast<int>(warp); i < pf; i += issuers_for<STAGES>()) {
      if constexpr (KBS == 1) tma_prefetch_l2_2d(&tmW, (kb_begin + i) * kBK, n0);
      else tma_prefetch_l2_3d(&tmW, 0, n0, kb_begin + i * KBS);
    }
  }
  // Global memory (operands, scales, y) is read or written only after the
  // preceding grids of the stream have completed; the set-up above overlaps
  // their tail.  Tensor memory is allocated only after the wait, so this CTA
  // never holds it while it waits for another grid.
  griddep_wait();
  if (warp == kMmaWarp) {
    tmem_alloc(holder_addr, C::kTmemCols);
    tmem_relinquish();
  }
  if (!REALIGN && lane == 0 && warp < 4) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *holder;
  // Our dependents may launch once every CTA of this grid holds its tensor
  // memory: a dependent CTA sharing an SM can then only wait for ours to
  // free it, never take it first.
  griddep_launch_dependents();
  const WaitCtx wc{p.err, abort_flag, p.budget_ns};

  if (warp < 4) {
    // ------------------------------------------------------------ producer
    if (!REALIGN) {
      // Stage s is filled by warp s % kIssuers (lane 0): a single issuing
      // thread cannot keep enough TMA copies in flight to stream the weight.
      // Each stage has one owner, which therefore reuses it in order.
      constexpr int kIssuers = issuers_for<STAGES>();
      if (lane == 0 && static_cast<int>(warp) < kIssuers) {
        const uint64_t pol_stream = l2_policy_evict_first();
        const uint64_t pol_keep = l2_policy_evict_last();
        int last_use[STAGES];
        for (int s = 0; s < STAGES; ++s) last_use[s] = -1;
        for (int i = static_cast<int>(warp); i < my_it; i += kIssuers) {
          const int stage = i % STAGES;
          const uint32_t use = static_cast<uint32_t>(i / STAGES);
          if (!mbar_wait_bounded(empty_bar(stage), (use & 1u) ^ 1u, wc, kErrWaitProducer)) break;
          mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
          const int kb = kb_begin + i * KBS;
          if constexpr (KBS == 1) {
            tma_load_2d_hint(sA(stage), &tmW, full_bar(stage), kb * kBK, n0, pol_stream);
            tma_load_2d_hint(sB(stage), &tmX, full_bar(stage), kb * kBK, 0, pol_keep);
          } else {
            tma_load_3d_hint(sA(stage), &tmW, full_bar(stage), 0, n0, kb, pol_stream);
            tma_load_3d_hint(sB(stage), &tmX, full_bar(stage), 0, 0, kb, pol_keep);
          }
          last_use[stage] = static_cast<int>(use);
        }
        for (int s = 0; s < STAGES; ++s)
          if (last_use[s] >= 0)
            drain_wait(full_bar(s), static_cast<uint32_t>(last_use[s]) & 1u, p.err, p.budget_ns);
      }
      __syncwarp();
    } else {
      const int ptid = static_cast<int>(threadIdx.x);
      uint32_t stage = 0, phase = 0;
      for (int kb = kb_begin; kb < kb_end; ++kb) {
        // all of this K block's loads (w rows and x rows) are issued before
        // the first is used, so the block costs one memory latency
        RealignRegs<kBN, 128> ga;
        RealignRegs<MP, 128> gb;
        realign_load(ga, p.w, p.N, p.K, n0, kb * kBK, ptid);
        realign_load(gb, p.x, p.M, p.K, 0, kb * kBK, ptid);
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, wc, kErrWaitProducer)) break;
        realign_store(sA(stage), ga, ptid);
        realign_store(sB(stage), gb, ptid);
        fence_proxy_async_smem();
        mbar_arrive(full_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }

    // ------------------------------------------------------------ partials
    // TMEM lane = n within the tile, column = m.  Park them in shared memory
    // as part[m][n] so the cluster reduction reads 16-byte runs along n.
    // The scale of column n is fetched now, its latency hidden behind the
    // last MMAs, and staged in shared memory for the reduction.
    const uint32_t n_local = warp * 32u + lane;
    const float my_scale =
        n0 + static_cast<int>(n_local) < p.N ? __ldg(p.scale + n0 + n_local) : 0.f;
    const bool have_acc = (my_kb == 0) || mbar_wait_bounded(acc_full_bar, 0u, wc, kErrWaitEpilogue);
    scale_s[n_local] = my_scale;
    if (have_acc && direct) {
      // lane = output channel n, TMEM column = token m: y[m][n] for the
      // warp's 32 channels, one coalesced 64-byte row segment per m
      tc_fence_after_sync();
      const int n = n0 + static_cast<int>(n_local);
#pragma unroll 1
      for (int c = 0; c < MP / 32; ++c) {
        uint32_t v[32];
        if (my_kb > 0) {
          tmem_ld_32x32b_x32(tmem_base + ((warp * 32u) << 16) + c * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = c * 32 + j;
            if (m < p.M)
              p.y[static_cast<size_t>(m) * static_cast<size_t>(p.N) + n] = static_cast<uint16_t>(
                  pack_bf16x2(__uint_as_float(v[j]) * my_scale, 0.f) & 0xFFFFu);
          }
        }
      }
    } else if (have_acc) {
      tc_fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < MP / 32; ++c) {
        uint32_t v[32];
        if (my_kb > 0) {
          tmem_ld_32x32b_x32(tmem_base + ((warp * 32u) << 16) + c * 32, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
          sts_f32(part + static_cast<uint32_t>(((c * 32 + j) * kBN + n_local) * 4),
                  __uint_as_float(v[j]));
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_e4m3_f32(kBN, MP);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int i = 0; i < my_it; ++i) {
        if (!mbar_wait_bounded(full_bar(stage), phase, wc, kErrWaitMma)) {
          ok = false;
          break;
        }
        // TMA data reach the MMA through the full barrier alone; operands written
        // by producer threads (generic proxy) additionally need the tcgen05 fence
        if (REALIGN) tc_fence_after_sync();
#pragma unroll
        for (int j = 0; j < KBS; ++j) {
          const uint64_t a_desc = sdesc_kmajor_sw128(sA(stage) + j * C::kABytes1);
          const uint64_t b_desc = sdesc_kmajor_sw128(sB(stage) + j * C::kBBytes1);
#pragma unroll
          for (int k = 0; k < kBK / kMmaK; ++k)
            tc_mma_f8(tmem_base, a_desc + 2u * k, b_desc + 2u * k, kIdesc,
                      (i > 0 || j > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(empty_bar(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && my_kb > 0) tc_commit(acc_full_bar);
      tc_commit(mma_done_bar);
      drain_wait(mma_done_bar, 0u, p.err, p.budget_ns);
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- reduce
  // Every CTA of the cluster has parked its partials; each now reduces an
  // equal share of the M x 128 outputs of this n-tile, reading all partials
  // through distributed shared memory, and stores scaled bf16.  A thread
  // takes two float4 groups at a time and issues all their remote loads
  // before it sums any, so each round pays one remote latency.
  tc_fence_before_sync();
  if (!direct) {
    cluster_sync_all();
    const int groups = p.M * (kBN / 4);  // float4 groups of valid rows
    const int g_begin = static_cast<int>((static_cast<long long>(groups) * rank) / splits);
    const int g_end = static_cast<int>((static_cast<long long>(groups) * (rank + 1)) / splits);
    auto finish = [&](int g, const float4* v) {
      float4 s = v[0];  // summed in split order
#pragma unroll
      for (int q = 1; q < kMaxSplits; ++q) {
        if (q < splits) {
          s.x += v[q].x;
          s.y += v[q].y;
          s.z += v[q].z;
          s.w += v[q].w;
        }
      }
      const int m = g / (kBN / 4);
      const int nl = (g % (kBN / 4)) * 4;
      const float4 sc = *reinterpret_cast<const float4*>(scale_s + nl);
      const int n = n0 + nl;
      uint16_t* yr = p.y + static_cast<size_t>(m) * static_cast<size_t>(p.N);
      const uint32_t lo = pack_bf16x2(s.x * sc.x, s.y * sc.y);
      const uint32_t hi = pack_bf16x2(s.z * sc.z, s.w * sc.w);
      if (n + 4 <= p.N && p.vec_store) {
        *reinterpret_cast<uint2*>(yr + n) = make_uint2(lo, hi);
      } else {
        const uint16_t h[4] = {static_cast<uint16_t>(lo & 0xFFFFu), static_cast<uint16_t>(lo >> 16),
                               static_cast<uint16_t>(hi & 0xFFFFu), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n + j < p.N) yr[n + j] = h[j];
      }
    };
    auto group_off = [&](int g) {
      return part + static_cast<uint32_t>(((g / (kBN / 4)) * kBN + (g % (kBN / 4)) * 4) * 4);
    };
    for (int g0 = g_begin + static_cast<int>(threadIdx.x); g0 < g_end; g0 += 2 * kThreads) {
      const int g1 = g0 + kThreads;
      const bool two = g1 < g_end;
      const uint32_t off0 = group_off(g0);
      const uint32_t off1 = two ? group_off(g1) : off0;
      float4 v0[kMaxSplits], v1[kMaxSplits];
#pragma unroll
      for (int q = 0; q < kMaxSplits; ++q) {
        if (q < splits) {
          v0[q] = ld_dsmem_f32x4(mapa_shared(off0, static_cast<uint32_t>(q)));
          v1[q] = ld_dsmem_f32x4(mapa_shared(off1, static_cast<uint32_t>(q)));
        }
      }
      finish(g0, v0);
      if (two) finish(g1, v1);
    }
  }
  // nobody leaves while another CTA may still read its shared memory
  cluster_sync_all();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ------------------------------------------------------------------ dispatch
struct DEntry {
  int mp, stages;
  bool realign;
  int kbs;
  const void* fn;
  int smem;
};

template <int MP, int S, bool R, int KBS = 1>
DEntry make_dentry() {
  return DEntry{MP, S, R, KBS,
                reinterpret_cast<const void*>(&fp8_linear_decode_kernel<MP, S, R, KBS>),
                DCfg<MP, S, R, KBS>::kSmemBytes};
}

const DEntry kDEntries[] = {
    make_dentry<32, 2, false>(),  make_dentry<32, 3, false>(),  make_dentry<32, 4, false>(),
    make_dentry<32, 6, false>(),  make_dentry<32, 8, false>(),  make_dentry<32, 10, false>(),
    make_dentry<64, 2, false>(),  make_dentry<64, 3, false>(),  make_dentry<64, 4, false>(),
    make_dentry<64, 6, false>(),  make_dentry<64, 8, false>(),  make_dentry<128, 2, false>(),
    make_dentry<128, 4, false>(), make_dentry<256, 2, false>(), make_dentry<256, 3, false>(),
    make_dentry<256, 4, false>(), make_dentry<32, 3, true>(),   make_dentry<32, 4, true>(),
    make_dentry<64, 3, true>(),   make_dentry<64, 4, true>(),   make_dentry<128, 2, true>(),
    // several K blocks per stage (3-D boxes): one large copy of w per stage
    make_dentry<32, 2, false, 4>(), make_dentry<32, 4, false, 2>(), make_dentry<32, 5, false, 2>(),
    make_dentry<64, 2, false, 4>(), make_dentry<64, 4, false, 2>(), make_dentry<128, 3, false, 2>(),
    make_dentry<256, 2, false, 2>(),
};

const DEntry* dfind(int mp, int stages, bool realign, int kbs) {
  for (const DEntry& e : kDEntries)
    if (e.mp == mp && e.stages == stages && e.realign == realign && e.kbs == kbs) return &e;
  return nullptr;
}

}  // namespace

bool dec_config_supported(int mp, int stages, bool realign, int kbs) {
  return dfind(mp, stages, realign, kbs) != nullptr;
}

int dec_smem_bytes(int mp, int stages, bool realign, int kbs) {
  const DEntry* e = dfind(mp, stages, realign, kbs);
  return e ? e->smem : -1;
}

int dec_threads(bool) { return kThreads; }

int dec_tmem_cols(int mp) { return mp <= 32 ? 32 : (mp <= 64 ? 64 : (mp <= 128 ? 128 : 256)); }

int dec_stage_bytes(int mp, int kbs) { return (kBN + mp) * kBK * kbs; }

cudaError_t dec_prepare(int mp, int stages, bool realign, int kbs) {
  const DEntry* e = dfind(mp, stages, realign, kbs);
  if (!e) return cudaErrorInvalidValue;
  cudaError_t r =
      cudaFuncSetAttribute(e->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, e->smem);
  if (r != cudaSuccess) return r;
  // several decode CTAs share an SM: ask for the largest shared-memory
  // carveout, or the SM may be configured with room for only one of them
  return cudaFuncSetAttribute(e->fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

// Resident CTAs per SM, counted from the kernel's resources: shared memory
// (228 KB per SM, 1 KB of it reserved per CTA), registers (allocated per warp
// in units of 256), threads (2048 per SM) and the 32-CTA limit.
cudaError_t dec_blocks_per_sm(int mp, int stages, bool realign, int kbs, int* out) {
  const DEntry* e = dfind(mp, stages, realign, kbs);
  if (!e) return cudaErrorInvalidValue;
  cudaFuncAttributes fa;
  cudaError_t r = cudaFuncGetAttributes(&fa, e->fn);
  if (r != cudaSuccess) return r;
  const int smem = e->smem + static_cast<int>(fa.sharedSizeBytes) + 1024;
  const int by_smem = 233472 / smem;
  const int regs_per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
  const int warps = kThreads / 32;
  const int by_regs = regs_per_warp > 0 ? 65536 / (warps * regs_per_warp) : 32;
  const int by_threads = 2048 / kThreads;
  int n = by_smem < by_regs ? by_smem : by_regs;
  n = n < by_threads ? n : by_threads;
  *out = n < 32 ? n : 32;
  return cudaSuccess;
}

cudaError_t dec_max_active_clusters(int mp, int stages, bool realign, int kbs, int splits,
                                    int grid, int* out) {
  const DEntry* e = dfind(mp, stages, realign, kbs);
  if (!e) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(e->smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, e->fn, &cfg);
}

cudaError_t launch_decode(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                          const DecConfig& c, cudaStream_t s) {
  const DEntry* e = dfind(c.mp, c.stages, c.realign, c.kbs);
  if (!e) return cudaErrorInvalidValue;
  // every split must cover whole stages
  if (c.kbs > 1 && (a.num_kb % (c.splits * c.kbs)) != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c.n_tiles * c.splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(e->smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_pdl(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  CUtensorMap mA = tmA, mB = tmB;
  GemmArgs args = a;
  int splits = c.splits;
  void* params[] = {&mA, &mB, &args, &splits};
  return cudaLaunchKernelExC(&cfg, e->fn, params);
}

}  // namespace fp8g
