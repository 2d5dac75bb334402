// gemm_tc2.cu -- persistent tcgen05 kernel on CTA pairs (cta_group::2) for
// the scaled FP8 linear layer  y = bf16((x_e4m3 . w_e4m3^T, fp32 acc) * scale[n]).
//
// The pages' fastest Blackwell submission runs CUTLASS's two-SM UMMA tiles
// (256 x 256 x 128) for the large shapes ("claude-fable-5" page, CUTLASS 4.0
// SM100 paragraph).  This kernel is that idea written directly in PTX: a
// 2-CTA cluster owns a 256 x BN output tile; CTA r (r = 0, 1) loads x rows
// [256 mb + 128 r, +128) and w rows [BN nb + BN/2 r, +BN/2) of every 128-byte
// K block into its own shared memory, and the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256), which reads A and B from both CTAs and
// leaves accumulator rows 0-127 in CTA 0's TMEM and rows 128-255 in CTA 1's.
// Per SM this halves the B bytes held in shared memory and read by the
// tensor core, which is what limits the one-CTA 128-row tile.
//
// Roles per CTA: warps 0-3 epilogue (TMEM -> * scale -> bf16 -> swizzled
// shared-memory staging -> TMA store), warp 4 TMEM allocation (both CTAs)
// and MMA issue (even CTA, one thread), warps 5-8 TMA producers, one thread
// each: x of a stage's first K block, x of its second, w of its first, w of
// its second (a TMA copy keeps its issuing thread busy for about a hundred
// cycles, so one thread per operand cannot keep the tensor cores fed); with
// one 3-D box per operand and stage (K % 128 == 0) the two producers of an
// operand take alternate stages.  Short-K shapes use eight epilogue warps
// (0-7), the MMA warp 8 and three producers (9-11).
//
// A stage holds two 128-byte K blocks.  The issuing thread spends about 95
// cycles per tcgen05.mma and about 70 per barrier wait even when the stage
// is ready, so with one K block (4 MMAs, 512 tensor cycles at N = 256) per
// wait and commit, issue rather than the tensor core set the pace; with two
// (8 MMAs, 1024 cycles) per wait and commit it keeps ahead.
// Synchronisation:
//   full[s]   in CTA 0 only: CTA 0's producers of the stage arm it, each
//             with its box's bytes for both CTAs; both CTAs' loads complete
//             on it;
//   empty[s]  in both CTAs: the MMA commit multicasts to both;
//   tfull[a]  in both CTAs: multicast commit after a tile's last K block;
//   tempty[a] in CTA 0 only: every epilogue warp of the pair (8 or 16)
//             arrives on it.
// Every wait is bounded, as in the one-CTA kernel.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace fp8g {
namespace {

constexpr int kBK = 128;
constexpr int kKbPerStage = 2;  // 128-byte K blocks per pipeline stage
constexpr int kStgBytes = 2048;  // one 32 x 32 bf16 staging box (64-byte swizzle)
// tiles of at most this many K blocks (K <= 3072) take the rolled epilogue loop
constexpr int kRolledEpilogueMaxKb = 24;

// EPI epilogue warps (4, or 8 for short-K tiles where the epilogue, not the
// MMA, sets the pace: two warps per TMEM lane quarter, each storing half of
// the tile's columns), then the TMEM/MMA warp, then the TMA producer warps
// (x first K block, x second, w first, w second; w's two by one warp when
// there are eight epilogue warps).
template <int BN, int STAGES, int EPI = 4>
struct Cfg2 {
  static constexpr int kEpiWarps = EPI;
  static constexpr int kMmaWarp = EPI;
  static constexpr int kProdWarp0 = EPI + 1;
  // four TMA producer warps, or three with eight epilogue warps (the third
  // issues both of w's K blocks): twelve warps leave 168 registers a thread
  static constexpr int kNumProd = EPI == 8 ? 3 : 4;
  static constexpr int kThreads = 32 * (EPI + 1 + kNumProd);
  static constexpr int kChunks = BN / 32;
  // chunks [0, kSplit) belong to warps 0-3, [kSplit, kChunks) to warps 4-7
  static constexpr int kSplit = EPI == 8 ? (kChunks + 1) / 2 : kChunks;
  static constexpr int kABytes1 = 128 * kBK;       // this CTA's 128 rows of x, one K block
  static constexpr int kBRows = BN / 2;            // this CTA's rows of w
  static constexpr int kBBytes1 = kBRows * kBK;    // ... one K block
  static constexpr int kABytes = kKbPerStage * kABytes1;
  static constexpr int kBBytes = kKbPerStage * kBBytes1;
  static constexpr int kStageBytes = kABytes + kBBytes;  // [x kb0][x kb1][w kb0][w kb1]
  static constexpr int kTmemCols = (2 * BN <= 256) ? 256 : 512;
  static constexpr int kStgOff = STAGES * kStageBytes;  // EPI warps x kBoxes staging boxes
  static constexpr int kNumBars = 2 * STAGES + 6 + kEpiWarps;  // + one per epilogue warp
  // Staging boxes per epilogue warp: with eight warps, one per chunk of the
  // warp where shared memory allows (no chunk then waits for an earlier
  // store of the same tile to read its box), else two used in turn.
  static constexpr int kBoxes =
      (EPI == 8 && kSplit > 2 &&
       1024 + kStgOff + kEpiWarps * kSplit * kStgBytes + kEpiWarps * BN * 4 + kNumBars * 8 + 16 <=
           232448)
          ? kSplit
          : 2;
  // each epilogue warp's copy of the tile's BN scales, where it fits
  static constexpr int kScOff = kStgOff + kEpiWarps * kBoxes * kStgBytes;
  static constexpr bool kScInSmem =
      1024 + kScOff + kEpiWarps * BN * 4 + kNumBars * 8 + 16 <= 232448;
  static constexpr int kBarOff = kScOff + (kScInSmem ? kEpiWarps * BN * 4 : 0);
  static constexpr int kPartBytes = BN * 128;  // one warp's share of a partial sum (32 x BN fp32)
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8 + 16;
  static_assert(EPI == 4 || EPI == 8, "epilogue warps");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(kBRows % 8 == 0, "B half must be whole 8-row swizzle atoms");
  static_assert(kKbPerStage == 1 || kKbPerStage == 2, "K blocks per stage");
  static_assert(kKbPerStage == 2 || STAGES % 2 == 0, "one-K-block stages alternate producers");
  static_assert(kABytes1 % 1024 == 0 && kBBytes1 % 1024 == 0,
                "every K block of a stage must start on a 1024-byte swizzle atom");
  // the split tail and the last unit shared with the producers exist with
  // four epilogue warps only
  static_assert(EPI == 8 || kEpiWarps * kPartBytes <= STAGES * kStageBytes,
                "a partial sum must fit in the ring it reuses");
  // last unit: 8 warps x (up to) half the chunks, one staging box each
  static constexpr int kHalf = (BN / 32 + 1) / 2;
  static_assert(EPI == 8 || 2 * kEpiWarps * kHalf * kStgBytes <= STAGES * kStageBytes,
                "the last unit's staging boxes must fit in the ring");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

// Write one staged 32 x 32 chunk of y (lane l holds row row0 + l, columns
// col0 .. col0 + 31, as 16 packed bf16 pairs): one lane TMA-stores the box
// when every row of it is this tile's (rows past M are clipped by the
// store); when the box straddles the end of the tile's group, each lane
// stores its own row, if it is the group's, from registers.  A (possibly
// empty) bulk group is committed either way, so that staging-box accounting
// always refers to the same chunk.  Needs 16-byte y rows (vec_store).
__device__ __forceinline__ void emit_chunk(const CUtensorMap* tmY, uint32_t buf,
                                           const GemmArgs& p, int row0, int row_end, int col0,
                                           uint32_t lane, const uint32_t* packed) {
  const bool whole = row0 + 32 <= row_end || row_end >= p.M;
  if (lane == 0) {
    if (whole && row0 < p.M && col0 < p.N) tma_store_2d(tmY, buf, col0, row0);
    tma_store_commit();
  }
  if (!whole) {
    const int row = row0 + static_cast<int>(lane);
    if (row < row_end && row < p.M) {
      uint4* dst = reinterpret_cast<uint4*>(p.y + static_cast<size_t>(row) * p.N + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (col0 + 8 * q < p.N)
          dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                              packed[4 * q + 3]);
    }
  }
}

// Scale, round and store accumulator chunks [C0, C1) (32 columns each) of
// one warp's 32 rows: TMEM address t_row, y rows [row0, row0 + 32) of which
// those below row_end are the tile's, tile column block nb, scales from
// sc_s[column - nb BN] in shared memory (or, if sc_s is null, from
// scale[sbase + column]); chunk c is staged in box stg + (c - C0) *
// kStgBytes, which no earlier store uses.
template <int BN, int C0, int C1>
__device__ __forceinline__ void store_chunks(uint32_t t_row, uint32_t stg,
                                             const CUtensorMap* tmY, const GemmArgs& p,
                                             int row0, int row_end, int nb, int sbase,
                                             uint32_t lane, bool zero_acc, const float* sc_s) {
  static_assert(C0 < C1, "chunk range");
  float scv[C1 - C0];
#pragma unroll
  for (int c = C0; c < C1; ++c) {
    const int col = nb * BN + c * 32 + static_cast<int>(lane);
    scv[c - C0] = (sc_s == nullptr && col < p.N) ? __ldg(p.scale + sbase + col) : 0.f;
  }
  uint32_t va[32], vb[32];
  tmem_ld_32x32b_x32(t_row + C0 * 32, va);
#pragma unroll
  for (int c = C0; c < C1; ++c) {
    tmem_ld_wait();
    if (c + 1 < C1) {
      if ((c - C0) & 1) tmem_ld_32x32b_x32(t_row + (c + 1) * 32, va);
      else tmem_ld_32x32b_x32(t_row + (c + 1) * 32, vb);
    }
    const uint32_t* v = ((c - C0) & 1) ? vb : va;
    uint32_t packed[16];
    if (sc_s != nullptr) {
      const float4* scs = reinterpret_cast<const float4*>(sc_s + c * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 s4 = scs[j];
        const float a0 = zero_acc ? 0.f : __uint_as_float(v[4 * j]);
        const float a1 = zero_acc ? 0.f : __uint_as_float(v[4 * j + 1]);
        const float a2 = zero_acc ? 0.f : __uint_as_float(v[4 * j + 2]);
        const float a3 = zero_acc ? 0.f : __uint_as_float(v[4 * j + 3]);
        packed[2 * j] = pack_bf16x2(a0 * s4.x, a1 * s4.y);
        packed[2 * j + 1] = pack_bf16x2(a2 * s4.z, a3 * s4.w);
      }
    } else {
      const float sc = scv[c - C0];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float s0 = __shfl_sync(0xffffffffu, sc, 2 * j);
        const float s1 = __shfl_sync(0xffffffffu, sc, 2 * j + 1);
        const float a0 = zero_acc ? 0.f : __uint_as_float(v[2 * j]);
        const float a1 = zero_acc ? 0.f : __uint_as_float(v[2 * j + 1]);
        packed[j] = pack_bf16x2(a0 * s0, a1 * s1);
      }
    }
    const uint32_t buf = stg + static_cast<uint32_t>(c - C0) * kStgBytes;
    const uint32_t rb = buf + lane * 64u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      sts_v4(rb + ((static_cast<uint32_t>(q) ^ ((lane >> 1) & 3u)) << 4),
             make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]));
    fence_proxy_async_smem();
    __syncwarp();
    emit_chunk(tmY, buf, p, row0, row_end, nb * BN + c * 32, lane, packed);
  }
}

// ROLLED: the owner epilogue's chunk loop is rolled (two chunks per
// iteration) instead of fully unrolled; chosen for tiles of at most
// kRolledEpilogueMaxKb K blocks (see the loop).
template <int BN, int STAGES, bool ROLLED, int EPI>
__global__ void __launch_bounds__(Cfg2<BN, STAGES, EPI>::kThreads, 1)
    fp8_linear_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmY, const GemmArgs p,
                          const int num_m2_blk, const int num_n_blk, const int group_m) {
  using C = Cfg2<BN, STAGES, EPI>;
  static_assert(EPI == 4 || ROLLED, "eight epilogue warps use the rolled loop");
  constexpr int kEpiWarps = C::kEpiWarps;
  constexpr int kMmaWarp = C::kMmaWarp;
  constexpr int kProdWarp0 = C::kProdWarp0;
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
  auto part_bar = [&](uint32_t w) { return bar0 + 8u * (2 * STAGES + 5 + w); };
  // the epilogue warps' signal that the last unit's accumulator is complete
  const uint32_t last_bar = bar0 + 8u * (2 * STAGES + 5 + kEpiWarps);
  const uint32_t holder_addr = bar0 + 8u * C::kNumBars;
  volatile uint32_t* holder =
      reinterpret_cast<volatile uint32_t*>(gbase + C::kBarOff + 8 * C::kNumBars);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(gbase + C::kBarOff + 8 * C::kNumBars + 4);
  auto sA = [&](int s) { return sbase + static_cast<uint32_t>(s * C::kStageBytes); };
  auto sB = [&](int s) { return sbase + static_cast<uint32_t>(s * C::kStageBytes + C::kABytes); };
  // epilogue warp q's copy of the current tile's scales (when C::kScInSmem)
  auto sc_of = [&](uint32_t q) {
    return reinterpret_cast<float*>(gbase + C::kScOff + q * static_cast<uint32_t>(BN) * 4u);
  };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();  // 0 = even CTA (MMA issuer), 1 = its peer
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // CTA 0's producers of stage s: one per operand and K block, or one per
      // operand when a 3-D box carries both K blocks
      mbar_init(full_bar(s), kKbPerStage == 2 ? (p.kbox ? 2u : 4u) : 2u);
      mbar_init(empty_bar(s), 1u);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1u);
      mbar_init(tempty_bar(a), static_cast<uint32_t>(2 * kEpiWarps));
    }
    mbar_init(mma_done_bar, 1u);
    for (uint32_t w = 0; w < kEpiWarps; ++w) mbar_init(part_bar(w), 1u);
    mbar_init(last_bar, static_cast<uint32_t>(kEpiWarps));
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Both CTAs' barriers are initialised before any cross-CTA arrive or TMA
  // completion.
  cluster_sync_all();
  // Before the dependency wait, one producer per operand asks L2 for the
  // first stage of this pair's first tile (cp.async.bulk.prefetch.tensor): a
  // prefetch delivers nothing to the CTA and L2 is the point of coherence, so
  // the loads issued after the wait still observe every write of the
  // preceding grids.  The CTAs of a call become resident 1-3 us before the
  // previous call's grid completes, and after the wait all of them used to
  // ask DRAM for ~9 MB of first stages at once (first operands 2.4-3.7 us
  // after the wait; globaltimer stamps, 4096^3).  One stage: square 45.0 ->
  // 44.5 us, MLP 261.4 -> 260.5 us, 8192x8192x128 43.5 -> 42.9 us; two stages
  // gained no more.  The tile comes from the plain raster, so grouped layers
  // (whose tile map reads group offsets from memory) and split tails skip it.
  if (p.group_offsets == nullptr && p.tail_workers == 0 && p.num_kb > 0 && warp >= kProdWarp0 &&
      lane == 0 && ((warp - kProdWarp0) & 1u) == 0u && pair < num_m2_blk * num_n_blk) {
    const bool is_a = (warp - kProdWarp0) < 2u;
    int mb, nb;
    tile_coords(pair, num_m2_blk, num_n_blk, group_m, mb, nb);
    const int row =
        is_a ? mb * 256 + static_cast<int>(rank) * 128 : nb * BN + static_cast<int>(rank) * C::kBRows;
    const CUtensorMap* map = is_a ? &tmA : &tmB;
    if (EPI == 4 && p.kbox) {
      tma_prefetch_l2_3d(map, 0, row, 0);
    } else {
      tma_prefetch_l2_2d(map, 0, row);
      if (p.num_kb > 1) tma_prefetch_l2_2d(map, kBK, row);
    }
  }
  // Global memory (operands, scales, y) is touched only after the preceding
  // grids of the stream have completed; the set-up above overlaps their tail.
  // Tensor memory is allocated only after the wait, so this CTA never holds
  // it while it waits for another grid.
  griddep_wait();
  if (warp == kMmaWarp) {
    tmem_alloc_pair(holder_addr, C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kProdWarp0 && lane == 0) tma_prefetch_desc(&tmA);
  if (warp == kProdWarp0 + 2 && lane == 0) tma_prefetch_desc(&tmB);
  if (warp == 0 && lane == 0 && p.vec_store) tma_prefetch_desc(&tmY);
  // Both CTAs' tensor memory is allocated before any MMA or tcgen05.ld: every
  // thread arrives on a cluster barrier here; the MMA issuer and the epilogue
  // wait for it at once, the producers (no tensor memory until the last
  // unit) only after issuing their loads, so the first loads are in flight
  // while the allocation completes.  Our dependents may launch once every
  // CTA of this grid holds its tensor memory (each thread signals after its
  // wait): a dependent CTA sharing an SM can then only wait for ours to free
  // it, never take it first.
  tc_fence_before_sync();
  cluster_arrive_release();
  uint32_t tmem_base = 0;
  if (warp < kProdWarp0) {
    cluster_wait_acquire();
    tc_fence_after_sync();
    tmem_base = *holder;
    griddep_launch_dependents();
  }

  const WaitCtx wc{p.err, abort_flag, p.budget_ns};
  // a fresh mapper per role: each walks the tile list forward once
  auto mapper = [&]() {
    return TileMapper(p.group_offsets, p.groups, p.M, p.N, BN, num_n_blk, num_m2_blk, group_m);
  };
  const int num_tiles = static_cast<int>(mapper().total());
  const int num_kb = p.num_kb;
  const int tail_workers = p.tail_workers;

  if (warp >= kProdWarp0) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      const uint32_t q = warp - kProdWarp0;
      const bool is_a = q < 2;
      // two K blocks per stage: this thread loads K block `sub` of every
      // stage; one: it loads every other stage (those with it % 2 == sub).
      // With three producer warps the third loads both of w's K blocks.
      const int sub = static_cast<int>(q & 1u);
      const int half = kKbPerStage == 2 ? sub : 0;
      const int n_halves = (C::kNumProd == 3 && !is_a) ? 2 : 1;
      const CUtensorMap* map = is_a ? &tmA : &tmB;
      const uint32_t bytes = is_a ? C::kABytes1 : C::kBBytes1;
      const uint32_t off = is_a ? static_cast<uint32_t>(half * C::kABytes1)
                                : static_cast<uint32_t>(C::kABytes + half * C::kBBytes1);
      uint32_t it = 0;  // (unit, stage) iteration, shared numbering of all producers
      bool ok = true;
      WorkIter wi(pair, num_pairs, num_tiles, num_kb, tail_workers);
      WorkUnit wu;
      TileMapper tm = mapper();
      while (ok && wi.next(wu)) {
        const TileGeom tg = tm.at(wu.tile);
        const int row = is_a ? tg.row + static_cast<int>(rank) * 128
                             : tg.wrow + static_cast<int>(rank) * C::kBRows;
        for (int kb = wu.k0; kb < wu.k1; kb += kKbPerStage, ++it) {
          if (kKbPerStage == 1 && static_cast<int>(it & 1u) != sub) continue;
          if (EPI == 4 && p.kbox) {
            // one 3-D box carries both K blocks of this operand: the two
            // producers of an operand take alternate stages (a producer
            // never waits for a stage it does not load); a K block past the
            // unit's end is loaded but not used (past K: read as zero)
            if (static_cast<int>(it & 1u) != sub) continue;
            const uint32_t stage = it % STAGES;
            const uint32_t use = it / STAGES;
            if (!mbar_wait_bounded(empty_bar(stage), (use & 1u) ^ 1u, wc, kErrWaitProducer)) {
              ok = false;
              break;
            }
            const uint32_t box = is_a ? C::kABytes : C::kBBytes;
            if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2u * box);
            tma_load_3d_pair(sbase + stage * static_cast<uint32_t>(C::kStageBytes) +
                                 (is_a ? 0u : static_cast<uint32_t>(C::kABytes)),
                             map, mapa_shared(full_bar(stage), 0u), 0, row, kb);
            continue;
          }
          // An odd CTA's producer whose K block of this stage lies past the
          // unit's end (an odd number of K blocks) has nothing to load and
          // must not wait for the stage either: the MMA does not need it
          // there, so the stage could be released once more before the
          // producer looks, and a parity wait cannot tell those two phases
          // apart (it would wait for a completion that never comes).  The
          // even CTA's producer still arrives on the full barrier, which the
          // MMA waits for, so it can never fall that far behind.
          if (rank != 0 && kb + half >= wu.k1) continue;
          const uint32_t stage = it % STAGES;
          const uint32_t use = it / STAGES;
          if (!mbar_wait_bounded(empty_bar(stage), (use & 1u) ^ 1u, wc, kErrWaitProducer)) {
            ok = false;
            break;
          }
          for (int hh = 0; hh < n_halves; ++hh) {
            const int h = half + hh;
            const uint32_t o = off + static_cast<uint32_t>(hh) * bytes;
            if (kb + h < wu.k1) {
              if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2u * bytes);
              tma_load_2d_pair(sbase + stage * static_cast<uint32_t>(C::kStageBytes) + o, map,
                               mapa_shared(full_bar(stage), 0u), (kb + h) * kBK, row);
            } else if (rank == 0) {
              mbar_arrive(full_bar(stage));  // odd K-block count: this half stays empty
            }
          }
        }
      }
      // Teardown: every load this thread issued must have landed.  CTA 0
      // sees its full barriers complete; CTA 1's loads complete on CTA 0's
      // barrier, so it waits for the MMA's release of the stage instead.
      // Each stage barrier completes exactly one phase per use, so the last
      // use's parity is unambiguous.
      for (uint32_t back = 1; back <= STAGES && back <= it; ++back) {
        const uint32_t i = it - back;
        if (kKbPerStage == 1 && static_cast<int>(i & 1u) != sub) continue;
        const uint32_t ph = (i / STAGES) & 1u;
        if (rank == 0)
          drain_wait(full_bar(i % STAGES), ph, p.err, p.budget_ns);
        else
          drain_wait(empty_bar(i % STAGES), ph, p.err, p.budget_ns);
      }
    }
    __syncwarp();
    cluster_wait_acquire();  // the allocation barrier (see above)
    tc_fence_after_sync();
    tmem_base = *holder;
    griddep_launch_dependents();
    // ---- the last unit's epilogue is exposed (nothing overlaps it), so the
    // four producer warps, idle by then, store the second half of its chunks
    // for the 32 rows of their TMEM lane quarter (warp % 4); the epilogue
    // warps store the first half.  Only for a plain owned tile with a y map.
    {
      WorkIter wl(pair, num_pairs, num_tiles, num_kb, tail_workers);
      WorkUnit u, lu;
      int n_units = 0;
      while (wl.next(u)) {
        lu = u;
        ++n_units;
      }
      if (EPI == 4 && n_units > 0 && lu.owner && lu.q_end == pair + 1 && p.vec_store) {
        // the epilogue warps arrive once they have seen the last accumulator
        // complete (a parity wait on tfull itself could not tell its uses apart)
        if (mbar_wait_bounded(last_bar, 0u, wc, kErrWaitEpilogue)) {
          tc_fence_after_sync();
          TileMapper tm = mapper();
          const TileGeom tg = tm.at(lu.tile);
          const uint32_t quarter = warp & 3u;
          const uint32_t acc = static_cast<uint32_t>(n_units - 1) & 1u;
          const int row0 = tg.row + static_cast<int>(rank) * 128 + static_cast<int>(quarter) * 32;
          const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + acc * BN;
          const uint32_t stg = sbase + (kEpiWarps + (warp - kProdWarp0)) * C::kHalf * kStgBytes;
          // the scales were staged by epilogue warp `quarter` before it
          // arrived on last_bar
          store_chunks<BN, C::kHalf, C::kChunks>(t_row, stg, &tmY, p, row0, tg.row_end, tg.nb,
                                              tg.sbase, lane, num_kb == 0,
                                              C::kScInSmem ? sc_of(quarter) : nullptr);
          if (lane == 0) tma_store_wait_read<0>();
          __syncwarp();
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t kIdesc = idesc_e4m3_f32(256, BN);
      // descriptors of stage 0; stage s adds s * kStageBytes to the 16-byte
      // start-address field (shared addresses stay below 2^18, no carry out)
      const uint64_t a_desc0 = sdesc_kmajor_sw128(sA(0));
      const uint64_t b_desc0 = sdesc_kmajor_sw128(sB(0));
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      bool ready = false;  // full[stage] already seen complete (tested during the last issue)
      WorkIter wi(pair, num_pairs, num_tiles, num_kb, tail_workers);
      WorkUnit wu;
      while (ok && wi.next(wu)) {
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, wc, kErrWaitMma)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = wu.k0; kb < wu.k1; kb += kKbPerStage) {
          if (!ready && !mbar_wait_bounded(full_bar(stage), phase, wc, kErrWaitMma)) {
            ok = false;
            break;
          }
          // the TMA bytes reach the MMA through the full barrier alone: no tcgen05
          // fence per stage (one would hold the issue back until earlier MMAs drain)
          const uint32_t next = stage + 1 == STAGES ? 0u : stage + 1;
          const uint32_t next_phase = stage + 1 == STAGES ? phase ^ 1u : phase;
          ready = tc_mma_stage_pair(d_tmem, a_desc0 + stage * (C::kStageBytes >> 4),
                                    b_desc0 + stage * (C::kStageBytes >> 4), kIdesc,
                                    kb > wu.k0 ? 1u : 0u,
                                    (kKbPerStage == 2 && kb + 1 < wu.k1) ? 1u : 0u,
                                    C::kABytes1 >> 4, C::kBBytes1 >> 4, empty_bar(stage), 0x3,
                                    full_bar(next), next_phase);
          stage = next;
          phase = next_phase;
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull_bar(acc), 0x3);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      tc_commit_pair_mc(mma_done_bar, 0x1);
      drain_wait(mma_done_bar, 0u, p.err, p.budget_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Each warp owns 32 accumulator rows.  Per 32-column chunk: TMEM ->
    // registers, * scale[n], round to bf16, write the 32 x 32 box into one of
    // two 64-byte-swizzled staging boxes and let one lane TMA-store it (the
    // store clips rows >= M and columns >= N).  Without a usable y map
    // (N % 8 != 0 or y not 16-byte aligned) rows are stored directly.
    uint32_t acc = 0, acc_phase = 0, chunk_no = 0, part_phase = 0;
    const bool zero_acc = (num_kb == 0);
    const bool tma_y = p.vec_store != 0;
    const uint32_t stg =
        sbase + static_cast<uint32_t>(C::kStgOff) + warp * static_cast<uint32_t>(C::kBoxes * kStgBytes);
    constexpr int kChunks = BN / 32;
    // TMEM lane quarter (= tile rows) and chunk range of this warp: all
    // chunks of its quarter with four epilogue warps, half of them with eight
    const uint32_t quarter = warp & 3u;
    const int c_lo = warp < 4u ? 0 : C::kSplit;
    const int c_hi = warp < 4u ? C::kSplit : kChunks;
    // This warp's share of worker q's published partial sum: 32 rows x BN
    // columns stored [chunk][column][row], so that each store and load
    // instruction of the warp covers 128 contiguous bytes.
    constexpr int kPartFloats = kChunks * 32 * 32;
    const uint32_t slot = rank * 4u + warp;
    auto part_of = [&](int q) {
      return p.partials + (static_cast<size_t>(q) * 8u + slot) * kPartFloats;
    };
    WorkIter wi(pair, num_pairs, num_tiles, num_kb, tail_workers);
    WorkUnit wu;
    TileMapper tm = mapper();
    while (wi.next(wu)) {
      WorkIter peek = wi;
      WorkUnit nxt;
      const bool last = !peek.next(nxt);
      const TileGeom tg = tm.at(wu.tile);
      const int nb = tg.nb;
      const int row0 = tg.row + static_cast<int>(rank) * 128 + static_cast<int>(quarter) * 32;
      const int row = row0 + static_cast<int>(lane);
      const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + acc * BN;
      // TMEM -> registers double buffered: chunk c+1 is in flight while chunk c
      // is used (its registers are read only after the next tcgen05.wait::ld)
      uint32_t va[32], vb[32];
      // An owner's scales (lane l: column l of every chunk) are fetched before
      // its accumulator is ready, then copied to this warp's shared array so
      // that each chunk reads them as four-float broadcasts.
      float scv[kChunks];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int col = nb * BN + c * 32 + static_cast<int>(lane);
        scv[c] = (wu.owner && col < p.N) ? __ldg(p.scale + tg.sbase + col) : 0.f;
      }
      float* const sc_s = sc_of(warp);
      auto stage_scales = [&]() {
        if constexpr (C::kScInSmem) {
#pragma unroll
          for (int c = 0; c < kChunks; ++c) sc_s[c * 32 + lane] = scv[c];
          __syncwarp();
        }
      };
      if (EPI == 4 && last && wu.owner && wu.q_end == pair + 1 && tma_y) {
        // ---- the last unit, shared with the producer warps (see there): the
        // operand ring is idle, each chunk gets its own staging box in it
        if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, wc, kErrWaitEpilogue)) break;
        tc_fence_after_sync();
        stage_scales();
        if (lane == 0) mbar_arrive(last_bar);
        store_chunks<BN, 0, C::kHalf>(t_row, sbase + warp * C::kHalf * kStgBytes, &tmY, p, row0,
                                      tg.row_end, nb, tg.sbase, lane, zero_acc,
                                      C::kScInSmem ? sc_s : nullptr);
      } else if (!wu.owner) {
        // ---- a segment that does not hold the tile's first K block: publish
        // its fp32 partial sum for the owner
        if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, wc, kErrWaitEpilogue)) break;
        tc_fence_after_sync();
        float* dst = part_of(pair) + lane;
        tmem_ld_32x32b_x32(t_row, va);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          tmem_ld_wait();
          if (c + 1 < kChunks) {
            if (c & 1) tmem_ld_32x32b_x32(t_row + (c + 1) * 32, va);
            else tmem_ld_32x32b_x32(t_row + (c + 1) * 32, vb);
          }
          const uint32_t* v = (c & 1) ? vb : va;
#pragma unroll
          for (int j = 0; j < 32; ++j) __stcg(dst + (c * 32 + j) * 32, __uint_as_float(v[j]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_u64(p.flags + static_cast<size_t>(pair) * 8u + slot, p.epoch);
      } else {
        // ---- the tile's owner: own accumulator (+ the partial sums of
        // workers pair+1 .. q_end-1, in that order) * scale -> bf16 -> y
        if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, wc, kErrWaitEpilogue)) break;
        tc_fence_after_sync();
        stage_scales();
        // The partial sum of the first contributor is brought into shared
        // memory with one bulk copy: a tile with contributors is always its
        // owner's last unit, so the operand ring is idle (every MMA of the
        // pair has completed) and holds it.  Any further contributor (the
        // ranges hold at least half a tile, so at most one more) is read from L2.
        bool have_parts = true;
        const bool staged = wu.q_end > pair + 1;
        if (staged) {
          if (lane == 0) {
            for (int q = pair + 1; q < wu.q_end && have_parts; ++q)
              have_parts = flag_wait_bounded(p.flags + static_cast<size_t>(q) * 8u + slot,
                                             p.epoch, p.err, abort_flag, p.budget_ns);
            if (have_parts) {
              fence_proxy_async_global();
              mbar_arrive_expect_tx(part_bar(warp), C::kPartBytes);
              bulk_load_g2s(sbase + warp * C::kPartBytes, part_of(pair + 1), C::kPartBytes,
                            part_bar(warp));
            }
          }
          have_parts = __shfl_sync(0xffffffffu, have_parts ? 1 : 0, 0) != 0;
          if (have_parts)
            have_parts = mbar_wait_bounded(part_bar(warp), part_phase, wc, kErrWaitPartial);
          part_phase ^= 1u;
        }
        const int q_end = have_parts ? wu.q_end : pair + 1;
        const float* staged_part =
            reinterpret_cast<const float*>(gbase + warp * C::kPartBytes) + lane;
        uint16_t* yrow = p.y + static_cast<size_t>(row) * static_cast<size_t>(p.N);
        if constexpr (ROLLED) {
          // Short tiles (the epilogue, not the MMA, tends to set the pace): a
          // rolled loop over chunk pairs (va, vb ping-pong) reuses the same
          // instructions for every pair of chunks; fully unrolled, each chunk
          // is new code that misses the instruction cache.  On long tiles the
          // epilogue hides behind the next tile's MMAs and either loop does
          // (rolling them too moved those shapes by under 1%).
          // one chunk: (partials added) * scale -> bf16 -> staged box -> TMA store
          // a chunk's (partials added) * scale -> bf16, into packed
          auto compute = [&](int c, const uint32_t (&v)[32], uint32_t (&packed)[16]) {
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = zero_acc ? 0.f : __uint_as_float(v[j]);
            if (q_end > pair + 1) {
#pragma unroll
              for (int j = 0; j < 32; ++j) a[j] += staged_part[(c * 32 + j) * 32];
            }
            for (int q = pair + 2; q < q_end; ++q) {
              const float* src = part_of(q) + c * 1024 + lane;
#pragma unroll
              for (int j = 0; j < 32; ++j) a[j] += __ldcg(src + j * 32);
            }
            if constexpr (C::kScInSmem) {
              const float4* scs = reinterpret_cast<const float4*>(sc_s + c * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 s4 = scs[j];
                packed[2 * j] = pack_bf16x2(a[4 * j] * s4.x, a[4 * j + 1] * s4.y);
                packed[2 * j + 1] = pack_bf16x2(a[4 * j + 2] * s4.z, a[4 * j + 3] * s4.w);
              }
            } else {
              const float sc = scv[c];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float s0 = __shfl_sync(0xffffffffu, sc, 2 * j);
                const float s1 = __shfl_sync(0xffffffffu, sc, 2 * j + 1);
                packed[j] = pack_bf16x2(a[2 * j] * s0, a[2 * j + 1] * s1);
              }
            }
          };
          // row `lane`, 16-byte chunk q at q ^ ((row >> 1) & 3): the 64-byte swizzle
          auto put = [&](uint32_t buf, const uint32_t (&packed)[16]) {
            const uint32_t rb = buf + lane * 64u;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              sts_v4(rb + ((static_cast<uint32_t>(q) ^ ((lane >> 1) & 3u)) << 4),
                     make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                packed[4 * q + 3]));
          };
          auto direct = [&](int c, const uint32_t (&packed)[16]) {
            const int col0 = nb * BN + c * 32;
            if (row < p.M && row < tg.row_end) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (col0 + j < p.N)
                  yrow[col0 + j] = static_cast<uint16_t>((j & 1) ? (packed[j >> 1] >> 16)
                                                                 : (packed[j >> 1] & 0xFFFFu));
              }
            }
          };
          if constexpr (C::kBoxes >= C::kSplit) {
            // Every chunk of the warp has its own box, so only the previous
            // tile's stores (issued a whole tile ago) must have read theirs
            // before this tile's first chunk is staged; each pair of chunks
            // is stored as soon as it is staged (storing all of them at the
            // end, behind one proxy fence, or a pair through one 32 x 64 box
            // with the 128-byte swizzle, was no faster).  A box straddling
            // the end of the tile's group is stored row by row from
            // registers instead.
            const bool whole = row0 + 32 <= tg.row_end || tg.row_end >= p.M;
            if (tma_y && chunk_no > 0) {
              if (lane == 0) tma_store_wait_read<0>();
              __syncwarp();
            }
            auto stage = [&](int c, const uint32_t (&packed)[16]) {
              if (tma_y && whole) put(stg + static_cast<uint32_t>(c - c_lo) * kStgBytes, packed);
              else direct(c, packed);
            };
            // proxy fence, then the TMA stores of staged chunks [c0, c1)
            auto flush = [&](int c0, int c1) {
              if (!tma_y) return;
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                for (int c = c0; c < c1; ++c) {
                  const int col0 = nb * BN + c * 32;
                  if (whole && row0 < p.M && col0 < p.N)
                    tma_store_2d(&tmY, stg + static_cast<uint32_t>(c - c_lo) * kStgBytes, col0,
                                 row0);
                }
                tma_store_commit();
              }
            };
            tmem_ld_32x32b_x32(t_row + c_lo * 32, va);
#pragma unroll 1
            for (int c = c_lo; c < c_hi; c += 2) {
              const bool two = c + 1 < c_hi;
              uint32_t pk0[16], pk1[16];
              tmem_ld_wait();
              if (two) tmem_ld_32x32b_x32(t_row + (c + 1) * 32, vb);
              compute(c, va, pk0);
              stage(c, pk0);
              if (two) {
                tmem_ld_wait();
                if (c + 2 < c_hi) tmem_ld_32x32b_x32(t_row + (c + 2) * 32, va);
                compute(c + 1, vb, pk1);
                stage(c + 1, pk1);
              }
              flush(c, two ? c + 2 : c + 1);
            }
            chunk_no += static_cast<uint32_t>(c_hi - c_lo);
          } else {
            // Chunks are handled in pairs (va, vb ping-pong): both are
            // computed, then staged in the warp's two boxes once the previous
            // pair's stores have read them, with one proxy fence for the two.
            tmem_ld_32x32b_x32(t_row + c_lo * 32, va);
#pragma unroll 1
            for (int c = c_lo; c < c_hi; c += 2) {
              const bool two = c + 1 < c_hi;
              uint32_t pk0[16], pk1[16];
              tmem_ld_wait();
              if (two) tmem_ld_32x32b_x32(t_row + (c + 1) * 32, vb);
              compute(c, va, pk0);
              if (two) {
                tmem_ld_wait();
                if (c + 2 < c_hi) tmem_ld_32x32b_x32(t_row + (c + 2) * 32, va);
                compute(c + 1, vb, pk1);
              }
              if (tma_y) {
                if (chunk_no > 0) {  // every earlier store has read its box
                  if (lane == 0) tma_store_wait_read<0>();
                  __syncwarp();
                }
                put(stg, pk0);
                if (two) put(stg + kStgBytes, pk1);
                fence_proxy_async_smem();
                __syncwarp();
                emit_chunk(&tmY, stg, p, row0, tg.row_end, nb * BN + c * 32, lane, pk0);
                if (two)
                  emit_chunk(&tmY, stg + kStgBytes, p, row0, tg.row_end, nb * BN + (c + 1) * 32,
                             lane, pk1);
              } else {
                direct(c, pk0);
                if (two) direct(c + 1, pk1);
              }
              chunk_no += two ? 2u : 1u;
            }
          }
        } else {
          tmem_ld_32x32b_x32(t_row, va);
#pragma unroll
          for (int c = 0; c < kChunks; ++c, ++chunk_no) {
            tmem_ld_wait();
            if (c + 1 < kChunks) {
              if (c & 1) tmem_ld_32x32b_x32(t_row + (c + 1) * 32, va);
              else tmem_ld_32x32b_x32(t_row + (c + 1) * 32, vb);
            }
            const uint32_t* v = (c & 1) ? vb : va;
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = zero_acc ? 0.f : __uint_as_float(v[j]);
            if (q_end > pair + 1) {
#pragma unroll
              for (int j = 0; j < 32; ++j) a[j] += staged_part[(c * 32 + j) * 32];
            }
            for (int q = pair + 2; q < q_end; ++q) {
              const float* src = part_of(q) + c * 1024 + lane;
#pragma unroll
              for (int j = 0; j < 32; ++j) a[j] += __ldcg(src + j * 32);
            }
            const int col0 = nb * BN + c * 32;
            uint32_t packed[16];
            if constexpr (C::kScInSmem) {
              const float4* scs = reinterpret_cast<const float4*>(sc_s + c * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 s4 = scs[j];
                packed[2 * j] = pack_bf16x2(a[4 * j] * s4.x, a[4 * j + 1] * s4.y);
                packed[2 * j + 1] = pack_bf16x2(a[4 * j + 2] * s4.z, a[4 * j + 3] * s4.w);
              }
            } else {
              const float sc = scv[c];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float s0 = __shfl_sync(0xffffffffu, sc, 2 * j);
                const float s1 = __shfl_sync(0xffffffffu, sc, 2 * j + 1);
                packed[j] = pack_bf16x2(a[2 * j] * s0, a[2 * j + 1] * s1);
              }
            }
            if (tma_y) {
              const uint32_t buf = stg + (chunk_no & 1u) * kStgBytes;
              if (chunk_no >= 2) {  // the store issued from this buffer two chunks ago
                if (lane == 0) tma_store_wait_read<1>();
                __syncwarp();
              }
              // row `lane`, 16-byte chunk q at q ^ ((row >> 1) & 3): the 64-byte swizzle
              const uint32_t rb = buf + lane * 64u;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                sts_v4(rb + ((static_cast<uint32_t>(q) ^ ((lane >> 1) & 3u)) << 4),
                       make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                  packed[4 * q + 3]));
              fence_proxy_async_smem();
              __syncwarp();
              emit_chunk(&tmY, buf, p, row0, tg.row_end, col0, lane, packed);
            } else if (row < p.M && row < tg.row_end) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (col0 + j < p.N)
                  yrow[col0 + j] = static_cast<uint16_t>((j & 1) ? (packed[j >> 1] >> 16)
                                                                 : (packed[j >> 1] & 0xFFFFu));
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0u));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    // every store must have finished reading shared memory before the CTA
    // exits (the writes themselves complete with the grid)
    if (tma_y && lane == 0) tma_store_wait_read<0>();
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  // The even CTA's MMAs (which write both CTAs' TMEM) are complete and every
  // epilogue has read its accumulators before the pair frees TMEM together.
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem_base, C::kTmemCols);
}

// ------------------------------------------------------------------ dispatch
struct Entry2 {
  int bn, stages, epi;
  const void* fn;         // unrolled owner epilogue loop (four epilogue warps only)
  const void* fn_rolled;  // rolled loop, for tiles of at most kRolledEpilogueMaxKb K blocks
  int smem, threads;
};

template <int BN, int S>
Entry2 make_entry2() {
  return Entry2{BN, S, 4, reinterpret_cast<const void*>(&fp8_linear_tc2_kernel<BN, S, false, 4>),
                reinterpret_cast<const void*>(&fp8_linear_tc2_kernel<BN, S, true, 4>),
                Cfg2<BN, S, 4>::kSmemBytes, Cfg2<BN, S, 4>::kThreads};
}

// Eight epilogue warps: rolled loop only, for short-K tiles.
template <int BN, int S>
Entry2 make_entry8() {
  const void* f = reinterpret_cast<const void*>(&fp8_linear_tc2_kernel<BN, S, true, 8>);
  return Entry2{BN, S, 8, f, f, Cfg2<BN, S, 8>::kSmemBytes, Cfg2<BN, S, 8>::kThreads};
}

const Entry2 kEntries2[] = {
    make_entry2<256, 3>(), make_entry2<224, 3>(), make_entry2<192, 3>(), make_entry2<160, 4>(),
    make_entry2<128, 4>(), make_entry8<256, 2>(), make_entry8<224, 3>(), make_entry8<192, 3>(),
    make_entry8<160, 3>(), make_entry8<128, 3>(),
};

const Entry2* find2(int bn, int stages, int epi) {
  for (const Entry2& e : kEntries2)
    if (e.bn == bn && e.stages == stages && e.epi == epi) return &e;
  return nullptr;
}

}  // namespace

bool tc2_config_supported(int bn, int stages, int epi) {
  return find2(bn, stages, epi) != nullptr;
}

int tc2_smem_bytes(int bn, int stages, int epi) {
  const Entry2* e = find2(bn, stages, epi);
  return e ? e->smem : -1;
}

int tc2_threads(int epi) { return epi == 8 ? 32 * 12 : 32 * 9; }

int tc2_max_stages(int bn, int smem_optin, int epi) {
  int best = 0;
  for (const Entry2& e : kEntries2)
    if (e.bn == bn && e.epi == epi && e.smem <= smem_optin && e.stages > best) best = e.stages;
  return best;
}

cudaError_t tc2_prepare(int bn, int stages, int epi) {
  const Entry2* e = find2(bn, stages, epi);
  if (!e) return cudaErrorInvalidValue;
  const cudaError_t r =
      cudaFuncSetAttribute(e->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, e->smem);
  if (r != cudaSuccess) return r;
  return cudaFuncSetAttribute(e->fn_rolled, cudaFuncAttributeMaxDynamicSharedMemorySize, e->smem);
}

cudaError_t tc2_max_active_pairs(int bn, int stages, int epi, int grid, int* out) {
  const Entry2* e = find2(bn, stages, epi);
  if (!e) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(e->threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(e->smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, e->fn_rolled, &cfg);
}

cudaError_t launch_tc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                       const GemmArgs& a, const TcConfig& c, cudaStream_t s) {
  const Entry2* e = find2(c.bn, c.stages, c.epi);
  if (!e || c.grid % 2) return cudaErrorInvalidValue;
  if (c.epi == 8 && (a.tail_workers > 0 || a.num_kb > kRolledEpilogueMaxKb))
    return cudaErrorInvalidValue;  // no split tail and no unrolled loop with eight warps
  const int num_m2 = (a.M + 255) / 256;
  const int num_n = (a.N + c.bn - 1) / c.bn;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(e->threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(e->smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_pdl(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  CUtensorMap mA = tmA, mB = tmB, mY = tmY;
  GemmArgs args = a;
  int m2 = num_m2, nn = num_n, gm = c.group_m;
  void* params[] = {&mA, &mB, &mY, &args, &m2, &nn, &gm};
  return cudaLaunchKernelExC(&cfg, a.num_kb <= kRolledEpilogueMaxKb ? e->fn_rolled : e->fn,
                             params);
}

}  // namespace fp8g
