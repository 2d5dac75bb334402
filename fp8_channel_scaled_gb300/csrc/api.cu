// api.cu -- the C ABI of include/fp8_gemm.h: argument validation, path
// selection, TMA descriptor encoding, launch, and the device error word.
//
// Path selection follows the regimes the pages' submissions pin instead of
// autotuning ("glm-5.2" page: dense tiles plus a skinny config for M <= 64;
// "claude-fable-5" page, Triton paragraph: split-K for M <= 64): M <= 64
// takes the split-K decode kernel, everything else the persistent tile
// kernel.  Rows that TMA cannot describe (pitch not a multiple of 16 bytes,
// or a base not 16-byte aligned) are first repitched into a workspace, or,
// without one, loaded by the in-kernel realigning producer.  Nothing derived
// from operand data is cached.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fp8_gemm.h"
#include "kernels.h"
#include "ptx.cuh"

namespace fp8g {
namespace {

// Device error word: kernels OR error bits into it; the host reads and clears
// it in fp8_gemm_check_device_error.
__device__ unsigned g_device_error_word;

// One thread waits for an mbarrier phase that nothing completes.
__global__ void selftest_wait_kernel(unsigned* err, unsigned long long budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1u);
  abort_flag = 0;
  fence_mbar_init();
  const WaitCtx wc{err, &abort_flag, budget_ns};
  (void)mbar_wait_bounded(b, 0u, wc, kErrWaitSelfTest);
}

constexpr int kMaxDevices = 64;
// Streams per device that keep a workspace; calls on further streams take
// theirs from the pool for the call.
constexpr int kStreamWorkspaces = 16;

struct StreamWorkspace {
  unsigned long long stream_id = 0;
  uint8_t* ptr = nullptr;
  size_t bytes = 0;
};
constexpr unsigned long long kDefaultBudgetNs = 1000000000ull;

struct DevState {
  bool init = false;
  int status = FP8GEMM_OK;
  int sm_count = 0;
  int smem_optin = 0;
  unsigned* err_word = nullptr;
  cudaMemPool_t pool = nullptr;  // private stream-ordered pool the shared workspace comes
  bool pool_failed = false;      // from; created on first use, never by the no-alloc entry
  void* noalloc_ws = nullptr;    // device address of g_noalloc_workspace on this device
  // Workspaces of the calls that bring none (repitch copies, split-tail
  // partial sums), one per stream: created on a stream's first need, grown
  // (in that stream's order) when a call needs more, kept until exit.  Calls
  // on one stream are ordered by the stream, so no two kernels that use the
  // same workspace ever overlap.  Streams are told apart by cudaStreamGetId,
  // which is never reused within a process.
  std::mutex ws_mu;
  StreamWorkspace ws[kStreamWorkspaces];
  int ws_count = 0;
  // Occupancy of each kernel configuration, queried once on first use so that
  // planning a call is plain arithmetic (-1: not queried yet, 0: cannot run).
  int tc2_pairs[6][3][2];        // [kTcTiles][kTc2Stages][epilogue warps 4, 8]: resident pairs
  int dec_blocks[4][7][2][3];       // [kDecMp][kDecStages][realign][kDecKbs]: CTAs per SM
  int dec_clusters[4][7][2][3][9];  // ... [splits]: resident clusters
  std::atomic<unsigned long long> calls{0};  // split-tail calls launched (epoch source)
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
unsigned long long g_budget_ns = 0;
unsigned g_last_error_bits = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

unsigned long long budget_ns() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_budget_ns == 0) {
    g_budget_ns = kDefaultBudgetNs;
    if (const char* s = std::getenv("FP8GEMM_WAIT_BUDGET_NS")) {
      const unsigned long long v = std::strtoull(s, nullptr, 10);
      if (v > 0) g_budget_ns = v;
    }
  }
  return g_budget_ns;
}

const int kTcTiles[] = {256, 224, 192, 160, 128, 64};  // 64: one-CTA tiles only
const int kTcStages[] = {3, 4, 5, 6, 7, 8, 9};
const int kTc2Stages[] = {2, 3, 4};
// Tiles of at most this many K blocks (K <= 1024) may take the pair kernel
// with eight epilogue warps: there the epilogue, not the MMA, sets the pace.
constexpr int kEpi8MaxKb = 8;
const int kDecMp[] = {32, 64, 128, 256};
const int kDecStages[] = {2, 3, 4, 5, 6, 8, 10};
const int kDecKbs[] = {1, 2, 4};  // 128-byte K blocks per decode stage

// Makes device `dev` current for the guard's lifetime and makes the caller's
// current device current again when it ends, so that no entry point leaves a
// different device current than it found (nothing is switched when `dev` is
// already current).
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      prev_ = -1;
    }
    if (prev_ == dev) {
      ok_ = true;
    } else if (cudaSetDevice(dev) == cudaSuccess) {
      ok_ = true;
      switched_ = prev_ >= 0;
    } else {
      cudaGetLastError();
    }
  }
  ~DeviceGuard() {
    if (switched_ && cudaSetDevice(prev_) != cudaSuccess) cudaGetLastError();
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = false;
  bool switched_ = false;
};

// Per-device set-up, once: properties, error word address, kernel attributes.
// It allocates nothing; the workspace pool is created on first pooled use.
// Device `dev` must be current (the callers hold a DeviceGuard).
int device_state(int dev, DevState** out) {
  if (dev < 0 || dev >= kMaxDevices) return FP8GEMM_EDEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  *out = &d;
  if (d.init) return d.status;
  d.init = true;
  std::memset(d.tc2_pairs, 0xff, sizeof(d.tc2_pairs));
  std::memset(d.dec_blocks, 0xff, sizeof(d.dec_blocks));
  std::memset(d.dec_clusters, 0xff, sizeof(d.dec_clusters));
  d.status = FP8GEMM_EDEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess) {
    cudaGetLastError();
    return d.status;
  }
  if (major != 10 || minor != 3) return d.status;  // the library is built for sm_103a only
  d.status = FP8GEMM_ELAUNCH;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err_word), g_device_error_word) !=
      cudaSuccess) {
    cudaGetLastError();
    return d.status;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      cudaGetLastError();
      return d.status;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  for (int bn : kTcTiles)
    for (int s : kTc2Stages)
      for (int epi : {4, 8})
        if (tc2_config_supported(bn, s, epi) && tc2_prepare(bn, s, epi) != cudaSuccess) {
          cudaGetLastError();
          return d.status;
        }
  for (bool r : {false, true}) {
    for (int bn : kTcTiles)
      for (int s : kTcStages)
        if (tc_config_supported(bn, s, r) && tc_prepare(bn, s, r) != cudaSuccess) {
          cudaGetLastError();
          return d.status;
        }
    for (int mp : kDecMp)
      for (int s : kDecStages)
        for (int kbs : kDecKbs)
          if (dec_config_supported(mp, s, r, kbs) && dec_prepare(mp, s, r, kbs) != cudaSuccess) {
            cudaGetLastError();
            return d.status;
          }
  }
  d.status = FP8GEMM_OK;
  return d.status;
}

// The device's private workspace pool, created on first use; nullptr if it
// cannot be created (calls then load unaligned rows in the kernel instead).
cudaMemPool_t workspace_pool(DevState& d, int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (d.pool || d.pool_failed) return d.pool;
  cudaMemPoolProps props;
  std::memset(&props, 0, sizeof(props));
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  if (cudaMemPoolCreate(&d.pool, &props) == cudaSuccess) {
    uint64_t keep = ~0ull;  // keep freed workspace memory for the next call
    cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
  } else {
    cudaGetLastError();
    d.pool = nullptr;
    d.pool_failed = true;
  }
  return d.pool;
}

// The workspace kept for stream `s` (id `sid`), grown to at least `need`
// bytes; nullptr in *out (and FP8GEMM_OK) when the device already keeps
// workspaces for kStreamWorkspaces other streams.  Growing frees the old
// block and takes the new one on `s`, i.e. after every earlier kernel of `s`,
// the only ones that used it.  The caller holds d.ws_mu until it has enqueued
// its kernels.  FP8GEMM_ENOMEM if the pool cannot provide the memory.
int stream_workspace(DevState& d, int dev, unsigned long long sid, size_t need, cudaStream_t s,
                     uint8_t** out) {
  *out = nullptr;
  StreamWorkspace* e = nullptr;
  for (int i = 0; i < d.ws_count; ++i)
    if (d.ws[i].stream_id == sid) e = &d.ws[i];
  if (!e) {
    if (d.ws_count == kStreamWorkspaces) return FP8GEMM_OK;
    e = &d.ws[d.ws_count++];
    e->stream_id = sid;
  }
  if (e->bytes < need) {
    cudaMemPool_t pool = workspace_pool(d, dev);
    if (!pool) return FP8GEMM_ENOMEM;
    if (e->ptr) {
      if (cudaFreeAsync(e->ptr, s) != cudaSuccess) cudaGetLastError();
      e->ptr = nullptr;
      e->bytes = 0;
    }
    // a quarter more than asked, in whole 2 MiB pages, so that a few
    // slightly larger calls do not each grow it
    const size_t grain = size_t(2) << 20;
    const size_t want = ((need + need / 4) + grain - 1) / grain * grain;
    void* p = nullptr;
    if (cudaMallocFromPoolAsync(&p, want, pool, s) != cudaSuccess || !p) {
      cudaGetLastError();
      return FP8GEMM_ENOMEM;
    }
    e->ptr = static_cast<uint8_t*>(p);
    e->bytes = want;
  }
  *out = e->ptr;
  return FP8GEMM_OK;
}

template <typename T, size_t n>
int index_of(const T (&arr)[n], T v) {
  for (size_t i = 0; i < n; ++i)
    if (arr[i] == v) return static_cast<int>(i);
  return -1;
}

// Resident CTA pairs of the pair kernel (bn, stages, epi) on the whole device.
int tc2_pairs(DevState& d, int bn, int stages, int epi) {
  const int i = index_of(kTcTiles, bn), j = index_of(kTc2Stages, stages);
  if (i < 0 || j < 0 || (epi != 4 && epi != 8)) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  int& v = d.tc2_pairs[i][j][epi == 8 ? 1 : 0];
  if (v < 0) {
    int pairs = 0;
    if (tc2_max_active_pairs(bn, stages, epi, d.sm_count & ~1, &pairs) != cudaSuccess) {
      cudaGetLastError();
      pairs = 0;
    }
    v = std::max(0, std::min(pairs, d.sm_count / 2));
  }
  return v;
}

// Resident decode CTAs per SM, or 0 if the configuration cannot run.  The
// tensor-memory budget (512 columns per SM) must cover every resident CTA, or
// a CTA's allocation would wait for another CTA to finish.
int dec_occupancy(DevState& d, int mp, int stages, bool realign, int kbs) {
  const int i = index_of(kDecMp, mp), j = index_of(kDecStages, stages), k = index_of(kDecKbs, kbs);
  if (i < 0 || j < 0 || k < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  int& v = d.dec_blocks[i][j][realign ? 1 : 0][k];
  if (v < 0) {
    v = 0;
    const int smem = dec_smem_bytes(mp, stages, realign, kbs);
    int blocks = 0;
    if (smem >= 0 && smem <= d.smem_optin) {
      if (dec_blocks_per_sm(mp, stages, realign, kbs, &blocks) != cudaSuccess) {
        cudaGetLastError();
        blocks = 0;
      }
      if (blocks * dec_tmem_cols(mp) <= 512) v = std::max(0, blocks);
    }
  }
  return v;
}

// Resident clusters of `splits` decode CTAs on the whole device.  Cluster
// placement (the CTAs of a cluster share a GPC) limits this below the per-SM
// count.  The query uses a grid large enough not to cap the answer.
int dec_clusters(DevState& d, int mp, int stages, bool realign, int kbs, int splits) {
  const int i = index_of(kDecMp, mp), j = index_of(kDecStages, stages), k = index_of(kDecKbs, kbs);
  if (i < 0 || j < 0 || k < 0 || splits < 1 || splits > 8) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  int& v = d.dec_clusters[i][j][realign ? 1 : 0][k][splits];
  if (v < 0) {
    int c = 0;
    if (dec_max_active_clusters(mp, stages, realign, kbs, splits, splits * 1024, &c) !=
        cudaSuccess) {
      cudaGetLastError();
      c = 0;
    }
    v = std::max(0, c);
  }
  return v;
}

// TMA descriptor of a byte matrix [rows, K] with row pitch `pitch` (a multiple
// of 16), box [box_rows, 128],
// 128-byte swizzle, out-of-bounds elements read as zero.
int encode_operand(CUtensorMap* map, const void* base, int rows, int K, size_t pitch,
                   int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8GEMM_OK : FP8GEMM_ELAUNCH;
}

// TMA descriptor of the same byte matrix viewed as [K / 128 blocks][rows][128
// bytes] (rows `pitch` bytes apart, K blocks 128 bytes apart; needs K % 128
// == 0 so that the view of each row ends at its last byte), with boxes of
// kbs K blocks x box_rows rows x 128 bytes and the 128-byte swizzle: one box
// lands as kbs consecutive K-major tiles of box_rows x 128 bytes.  Rows past
// `rows` read as zero.
int encode_operand_kblocks(CUtensorMap* map, const void* base, int rows, int K, size_t pitch,
                           int box_rows, int kbs) {
  const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / 128)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch), 128u};
  const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(kbs)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8GEMM_OK : FP8GEMM_ELAUNCH;
}

// TMA descriptor of y as bf16 [M, N] for 32 x 32 output boxes with the
// 64-byte swizzle (requires N % 8 == 0 and a 16-byte aligned y).
int encode_output(CUtensorMap* map, void* y, int M, int N) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2u};
  const cuuint32_t box[2] = {32u, 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, y, dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8GEMM_OK : FP8GEMM_ELAUNCH;
}

struct Plan {
  fp8gemm_plan pub;
  TcConfig tc;
  DecConfig dec;
  int Kp;                     // row pitch of the repitched operands
  bool rx, rw;                // x / w repitched into the workspace
  size_t x_off, w_off;        // offsets of the repitched x and w inside the workspace
  size_t part_off, flag_off;  // offsets of the split-tail partial sums and flags
};

// Tail workers per tail tile, at most.  A split tile's owner adds the other
// segments' partial sums (256 x BN x 4 bytes each) before it can write y; the
// pair kernel stages the first of them in shared memory and reads any further
// one from L2.  With twice as many workers as tail tiles every range is half a
// tile and a tile has two segments; with fewer (the pairs run out) the ranges
// no longer follow tile boundaries and a tile may have three.
constexpr int kTailWorkersPerTailTile = 2;

// CTA pairs that share the split tail of `tiles` tiles on `pairs` pairs, or
// 0 when splitting does not shorten the last wave.
int tail_workers_for(long long tiles, int pairs, int num_kb) {
  if (pairs <= 0 || num_kb <= 0) return 0;
  const long long rem = tiles % pairs;
  if (rem == 0) return 0;
  long long tw = std::min<long long>(pairs, rem * kTailWorkersPerTailTile);
  tw = std::min<long long>(tw, rem * num_kb);  // every range at least one K block
  return tw > rem ? static_cast<int>(tw) : 0;
}

// Whether the next kernel on `s` may be launched with programmatic stream
// serialization: always outside a stream capture; during one only when every
// node the launch will depend on is a kernel node, because a programmatic
// edge can only leave a kernel (after a copy, memset, event or memory node,
// e.g. a workspace allocation, the launch takes an ordinary edge).
bool pdl_ok(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaGraphNode_t* deps = nullptr;
  size_t n = 0;
  if (cudaStreamGetCaptureInfo(s, &cs, nullptr, nullptr, &deps, nullptr, &n) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (cs == cudaStreamCaptureStatusNone) return true;
  if (cs != cudaStreamCaptureStatusActive || n == 0 || !deps) return false;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(deps[i], &t) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (t != cudaGraphNodeTypeKernel) return false;
  }
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t v) { return (v + 255u) & ~static_cast<size_t>(255u); }

// Main path tile choice.  For each N tile (with the deepest ring that fits)
// and each tile kind -- one-CTA 128-row tiles or CTA-pair 256-row tiles --
// estimate waves x tile width, i.e. the wave quantisation of the persistent
// grid (a pair's 256 x BN tile takes about as long as one CTA's 128 x BN
// tile).  One-CTA tiles pay for the larger share of B each SM stages and
// reads (measured about 1.3x slower per tile); narrower tiles pay for their
// lower operand reuse.  The realigning producer exists for one-CTA tiles only.
int choose_tc(DevState& d, int M, int N, int num_kb, bool realign, bool can_split,
              const fp8gemm_options& o, TcConfig* out) {
  double best = 1e300;
  TcConfig pick{};
  for (int ctas : {2, 1}) {
    if (o.mma_ctas && ctas != o.mma_ctas) continue;
    if (ctas == 2 && realign) continue;
    for (int bn : kTcTiles) {
      if (o.tile_n && bn != o.tile_n) continue;
      int stages, units;
      if (ctas == 2) {
        if (o.epilogue_warps != 0 && o.epilogue_warps != 4 && o.epilogue_warps != 8)
          return FP8GEMM_EINVAL;
        const long long tiles = static_cast<long long>((M + 255) / 256) * ((N + bn - 1) / bn);
        // Eight epilogue warps for short-K tiles when every pair has at least
        // two tiles, so that epilogues overlap mainloops (8192 x 8192 x 128:
        // 64.5 -> 54.6 us, x 1024: 73.0 -> 67.4 us; with K = 2048 the two-stage
        // ring they leave room for is slower, 87.8 -> 104.8 us; one tile per
        // pair, 512 x 4096 x 1024: 8.3 -> 8.7 us).  No split tail with them.
        int epi = o.epilogue_warps;
        if (epi == 0) {
          const int pairs4 = tc2_pairs(d, bn, tc2_max_stages(bn, d.smem_optin, 4), 4);
          epi = (num_kb <= kEpi8MaxKb && !can_split && pairs4 > 0 && tiles >= 2LL * pairs4 &&
                 tc2_max_stages(bn, d.smem_optin, 8) > 0)
                    ? 8
                    : 4;
        }
        if (epi == 8 && (can_split || num_kb > 24)) continue;
        stages = o.stages ? o.stages : tc2_max_stages(bn, d.smem_optin, epi);
        if (stages == 0 || !tc2_config_supported(bn, stages, epi) ||
            tc2_smem_bytes(bn, stages, epi) > d.smem_optin)
          continue;
        const int pairs = tc2_pairs(d, bn, stages, epi);
        if (pairs <= 0) continue;
        // with a split tail the last wave costs its share of the tail's K
        // blocks plus the owners' reads of the other segments' partial sums
        const int tw = can_split ? tail_workers_for(tiles, pairs, num_kb) : 0;
        double waves;
        if (tw > 0) {
          const long long rem = tiles % pairs;
          waves = static_cast<double>(tiles / pairs) + static_cast<double>(rem) / tw +
                  0.05 * static_cast<double>(tw) / static_cast<double>(rem);
          units = pairs;
        } else {
          waves = static_cast<double>((tiles + pairs - 1) / pairs);
          units = static_cast<int>(std::min<long long>(tiles, pairs));
        }
        const double cost = waves * bn * (1.0 + 0.15 * (256 - bn) / 128.0);
        if (cost < best - 1e-9) {
          best = cost;
          pick = TcConfig{2, bn, stages, false, 2 * units, 16, tw, epi};
        }
      } else {
        stages = o.stages ? o.stages : tc_max_stages(bn, realign, d.smem_optin);
        if (stages == 0 || !tc_config_supported(bn, stages, realign) ||
            tc_smem_bytes(bn, stages, realign) > d.smem_optin)
          continue;
        const long long tiles = static_cast<long long>((M + 127) / 128) * ((N + bn - 1) / bn);
        units = static_cast<int>(std::min<long long>(tiles, d.sm_count));
        const long long waves = (tiles + d.sm_count - 1) / d.sm_count;
        const double cost =
            1.3 * static_cast<double>(waves) * bn * (1.0 + 0.15 * (256 - bn) / 128.0);
        if (cost < best - 1e-9) {
          best = cost;
          pick = TcConfig{1, bn, stages, realign, units, 16, 0, 4};
        }
      }
    }
  }
  if (!pick.bn) return FP8GEMM_EUNSUPPORTED;
  *out = pick;
  return FP8GEMM_OK;
}

int make_plan(DevState& d, const void* x, const void* w, int M, int N, int K,
              const fp8gemm_options* opt, Plan* pl) {
  fp8gemm_options o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (o.reserved != 0 || o.mma_ctas < 0 || o.mma_ctas > 2) return FP8GEMM_EINVAL;
  std::memset(pl, 0, sizeof(*pl));
  if (M == 0 || N == 0) return FP8GEMM_OK;  // nothing to do
  const size_t ldx = o.ldx ? o.ldx : static_cast<size_t>(K);
  const size_t ldw = o.ldw ? o.ldw : static_cast<size_t>(K);
  if (ldx < static_cast<size_t>(K) || ldw < static_cast<size_t>(K)) return FP8GEMM_EINVAL;
  // TMA reads an operand in place when its pitch is a multiple of 16 bytes and
  // its base 16-byte aligned (columns >= K then read as zero)
  const bool x_tma = (ldx % 16 == 0) && (!x || aligned16(x));
  const bool w_tma = (ldw % 16 == 0) && (!w || aligned16(w));
  const bool tma_ok = x_tma && w_tma;
  const bool contiguous = ldx == static_cast<size_t>(K) && ldw == static_cast<size_t>(K);
  // Operands TMA cannot tile are repitched into a workspace first, unless the
  // caller forbids it or asks for the in-kernel loader.  (On the decode path
  // too: the in-kernel loader holds its loads in registers and cannot keep
  // enough in flight; M = 32, N = 4096, K = 4127: 15.2 us repitched against
  // 21.4 us, N = K = 8191: 37.4 against 41.6 us.)
  const bool can_ws = !o.no_workspace;
  const bool repitch = K > 0 && !tma_ok && !o.force_realign && can_ws;
  // K == 0 has nothing to load; the realigning variant then issues no copy
  // and needs no tensor map.
  const bool realign = !repitch && (o.force_realign != 0 || !tma_ok || K == 0);
  int path = o.path;
  // M <= 64: the decode path.  Up to M = 192 it still wins while the weight
  // is at most 64 n-tiles of 128 rows (measured at N = 4096: M = 96 10.2 vs
  // 13.5 us, M = 128 10.2 vs 12.9 us, M = 160 11.1 vs 13.1 us, M = 192 11.8
  // vs 13.2 us; M = 256 13.2 vs 13.3 us; at N = 14336 the tile kernel is
  // faster).  129-192 rows run the decode kernel with x padded to 256 rows,
  // which is built for the TMA loader only.
  if (path == FP8GEMM_PATH_AUTO)
    path = (M <= 64 || (M <= 192 && N <= 64 * 128 && (M <= 128 || !realign)))
               ? FP8GEMM_PATH_DECODE
               : FP8GEMM_PATH_MAIN;
  if (path != FP8GEMM_PATH_MAIN && path != FP8GEMM_PATH_DECODE) return FP8GEMM_EINVAL;
  if (realign && K > 0 && !contiguous) return FP8GEMM_EALIGN;  // in-kernel loader needs pitch K
  pl->pub.path = path;
  pl->pub.realign = realign ? 1 : 0;
  pl->pub.repitch = repitch ? 1 : 0;
  pl->pub.launches = repitch ? 2 : 1;
  if (repitch) {
    // The copies' pitch is rounded up to 64 bytes, not just 16: with a pitch
    // that is an odd multiple of 16 every 128-byte K block of a row starts in
    // the middle of a 32-byte sector, and the GEMM slows down by a sixth
    // (4096 x 4096 x 4100 on operands padded to a 4112-byte pitch: 57.4 us
    // against 48.4 us at 4160 and 49.2 us at 4128; 2048 x 4096 x 4127: 28.5
    // us at 4128, 28.1 us at 4160).
    pl->Kp = (K + 63) & ~63;
    pl->rx = !x_tma;
    pl->rw = !w_tma;
    pl->x_off = 0;
    pl->w_off = pl->rx ? align256(static_cast<size_t>(M) * pl->Kp) : 0;
    pl->pub.workspace_bytes =
        pl->w_off + (pl->rw ? align256(static_cast<size_t>(N) * pl->Kp) : 0);
  }

  if (path == FP8GEMM_PATH_MAIN) {
    const int num_kb = (K + 127) / 128;
    int st = choose_tc(d, M, N, num_kb, realign, can_ws && o.split_tail && K > 0, o, &pl->tc);
    if (st != FP8GEMM_OK) return st;
    const bool pair = pl->tc.ctas == 2;
    if (pl->tc.tail_workers > 0) {
      // partial sums and flags of the split tail, after the repitch copies
      const size_t slots = static_cast<size_t>(pl->tc.tail_workers);
      pl->part_off = align256(pl->pub.workspace_bytes);
      pl->flag_off = pl->part_off + align256(slots * 2u * 128u * pl->tc.bn * sizeof(float));
      pl->pub.workspace_bytes = pl->flag_off + align256(slots * 8u * sizeof(unsigned long long));
      const long long tiles = static_cast<long long>((M + 255) / 256) * ((N + pl->tc.bn - 1) / pl->tc.bn);
      pl->pub.split_tiles = static_cast<int>(tiles % (pl->tc.grid / 2));
      pl->pub.tail_workers = pl->tc.tail_workers;
    }
    pl->pub.tile_m = pair ? 256 : 128;
    pl->pub.tile_n = pl->tc.bn;
    pl->pub.stages = pl->tc.stages;
    pl->pub.splits = 1;
    pl->pub.grid = pl->tc.grid;
    pl->pub.cluster = pair ? 2 : 1;
    pl->pub.threads = pair ? tc2_threads(pl->tc.epi) : tc_threads(realign);
    pl->pub.epilogue_warps = pair ? pl->tc.epi : 4;
    pl->pub.kblocks_per_stage = pair ? 2 : 1;
    pl->pub.smem_bytes = pair ? tc2_smem_bytes(pl->tc.bn, pl->tc.stages, pl->tc.epi)
                              : tc_smem_bytes(pl->tc.bn, pl->tc.stages, realign);
    pl->pub.occupancy = 1;  // one CTA per SM: the ring fills shared memory
    return FP8GEMM_OK;
  }

  // decode path: one cluster of `s` CTAs per 128-row n-tile, each CTA
  // streaming ceil(num_kb / s) K blocks.  How many clusters can be resident
  // at once is limited by cluster placement (CTAs of a cluster share a GPC),
  // not only by per-SM resources, so it is queried for each candidate.
  if (M > 256) return FP8GEMM_EUNSUPPORTED;
  const int num_kb = (K + 127) / 128;
  const int mp = M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256));
  const int n_tiles = (N + 127) / 128;
  int best_s = 0, best_stages = 0, best_occ = 0, best_kbs = 1;
  double best_cost = 1e300;
  // Up to 128 tokens over a weight of at least 8 MB with K % 256 == 0: two K
  // blocks per stage (3-D boxes), as many stages as fit one CTA per SM (5, 4
  // and 3 for x tiles of 32, 64 and 128 rows: ~200 KB of loads in flight)
  // and the most splits that keep every CTA on its own SM.  Measured back to
  // back against the single-K-block configurations the model below picks:
  // 32 x 8192 x 8192 13.8 against 14.5 us (2 splits), 32 x 14336 x 4096
  // 12.5 against 15.0 us (1 split, outputs stored straight from tensor
  // memory), 16 x 4096 x 4096 9.8 against 12.2 us, 64 x 4096 x 4096 8.7
  // against 10.2 us, 64 x 14336 x 4096 14.7 against 17.1 us, 128 x 8192 x
  // 8192 18.6 against 21.8 us; 64 x 8192 x 8192 16.1 against 15.9 us and 128
  // x 4096 x 4096 9.6 against 9.8 us are about even, 192 and 256 tokens gain
  // nothing and keep the model's choice.
  const int wide_stages = mp == 32 ? 5 : (mp == 64 ? 4 : (mp == 128 ? 3 : 0));
  const bool wide_auto = !o.tile_n && !o.stages && !o.splits && !realign && wide_stages > 0 &&
                         K % 256 == 0 && static_cast<long long>(N) * K >= (8LL << 20) &&
                         dec_config_supported(mp, wide_stages, false, 2);
  if (wide_auto) {
    const int occ = dec_occupancy(d, mp, wide_stages, false, 2);
    for (int sp = 8; sp >= 1 && occ > 0; sp /= 2) {
      if (num_kb % (2 * sp) != 0 || static_cast<long long>(n_tiles) * sp > d.sm_count) continue;
      if (dec_clusters(d, mp, wide_stages, false, 2, sp) * occ < n_tiles) continue;  // one wave
      best_s = sp;
      best_stages = wide_stages;
      best_occ = occ;
      best_kbs = 2;
      break;
    }
  }
  // Otherwise every configuration is costed by the model below.  Several K
  // blocks per stage (3-D boxes) need K % 128 == 0 (the boxes' view of a row
  // ends exactly at its last byte) and TMA-readable operands;
  // fp8gemm_options.tile_n selects the count on this path (0: automatic).
  if (o.tile_n && o.tile_n != 1 && o.tile_n != 2 && o.tile_n != 4) return FP8GEMM_EINVAL;
  for (int kbs : kDecKbs) {
    if (best_s) break;  // chosen above
    if (o.tile_n && kbs != o.tile_n) continue;
    if (kbs > 1 && (realign || K % 128 != 0)) continue;
  for (int stages : kDecStages) {
    if (o.stages && stages != o.stages) continue;
    if (!dec_config_supported(mp, stages, realign, kbs)) continue;
    const int occ = dec_occupancy(d, mp, stages, realign, kbs);
    if (occ <= 0) continue;
    const int s_max = std::max(1, std::min(8, num_kb / kbs));
    for (int s = 1; s <= s_max; ++s) {
      if (o.splits && s != o.splits) continue;
      if (kbs > 1 && num_kb % (s * kbs) != 0) continue;  // whole stages per split
      // cudaOccupancyMaxActiveClusters answers as if one CTA per SM (the same
      // count for every ring depth); clusters of CTAs that fit `occ` to an SM
      // do share SMs (4 splits x 4 stages, 64 clusters of 4 on 152 SMs, ran
      // in one wave), so the count scales with occ.
      const int clusters = dec_clusters(d, mp, stages, realign, kbs, s) * occ;
      if (clusters <= 0) continue;
      // The weight stream is shared by the SMs: a wave costs the K blocks of
      // its busiest SM (CTAs per SM x K blocks per CTA), more when some SMs
      // stay idle or an SM has less than ~160 KB of loads in flight, plus a
      // ramp of about five K blocks per wave and about one per split for the
      // cluster reduction.  (Calibrated on the 32 x 8192 x 8192 decode shape:
      // 4 splits x 4 stages, 256 CTAs two per SM, 15.2 us; 2 splits x 10
      // stages, 128 CTAs, 16.4 us; 4 splits x 8 stages, two waves, 21.1 us.)
      const long long waves = (n_tiles + clusters - 1) / clusters;
      const int per_cta = std::max((num_kb + s - 1) / s, 1);
      const long long grid = static_cast<long long>(std::min<long long>(n_tiles, clusters)) * s;
      const int per_sm = static_cast<int>((grid + d.sm_count - 1) / d.sm_count);
      const double coverage =
          static_cast<double>(std::min<long long>(grid, d.sm_count)) / d.sm_count;
      const double in_flight = static_cast<double>(per_sm) * stages *
                               dec_stage_bytes(mp, kbs) / (160.0 * 1024.0);
      double cost =
          static_cast<double>(waves) *
              (per_cta * per_sm * (1.0 + 0.5 * std::max(0.0, 1.0 - in_flight)) /
                   std::sqrt(coverage) +
               5.0) +
          1.0 * s;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best_s = s;
        best_stages = stages;
        best_occ = occ;
        best_kbs = kbs;
      }
    }
  }
  }
  if (best_s == 0) return FP8GEMM_EUNSUPPORTED;
  pl->dec.mp = mp;
  pl->dec.stages = best_stages;
  pl->dec.realign = realign;
  pl->dec.splits = best_s;
  pl->dec.n_tiles = n_tiles;
  pl->dec.kbs = best_kbs;
  pl->pub.tile_m = 128;
  pl->pub.tile_n = mp;
  pl->pub.stages = best_stages;
  pl->pub.splits = best_s;
  pl->pub.grid = n_tiles * best_s;
  pl->pub.cluster = best_s;
  pl->pub.threads = dec_threads(realign);
  pl->pub.smem_bytes = dec_smem_bytes(mp, best_stages, realign, best_kbs);
  pl->pub.kblocks_per_stage = best_kbs;
  pl->pub.occupancy = best_occ;
  return FP8GEMM_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return na && nb && pa < pb + nb && pb < pa + na;
}

// Device of a device-accessible allocation, or -1 for host / unknown memory.
int pointer_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return -1;
  return a.device;
}

// Enqueue the planned GEMM kernel.  xa / wa are the operands it reads (the
// caller's, or their repitched copies) with row pitch Ka.
// xa / wa (row pitches lxa / lwa) are the operands the kernel reads: the
// caller's, or their repitched copies; K is the true reduction length.
int launch_gemm(const Plan& pl, DevState& d, const void* xa, size_t lxa, const void* wa,
                size_t lwa, int K, const float* scale, void* y, int M, int N, uint8_t* ws,
                cudaStream_t s, const int* group_offsets = nullptr, int groups = 0) {
  GemmArgs a{};
  a.x = static_cast<const uint8_t*>(xa);
  a.w = static_cast<const uint8_t*>(wa);
  a.scale = scale;
  a.y = static_cast<uint16_t*>(y);
  a.M = M;
  a.N = N;
  a.K = K;  // the in-kernel loader (used only with pitch == K) reads rows of K bytes
  a.num_kb = (K + 127) / 128;
  a.vec_store = ((N % 8) == 0 && (reinterpret_cast<uintptr_t>(y) & 15u) == 0) ? 1 : 0;
  a.err = d.err_word;
  a.budget_ns = budget_ns();
  a.group_offsets = group_offsets;
  a.groups = groups;
  a.pdl = pdl_ok(s) ? 1 : 0;
  // a grouped layer's weight is [groups * N, K]
  const int w_rows = group_offsets ? groups * N : N;
  if (pl.pub.path == FP8GEMM_PATH_MAIN && pl.tc.tail_workers > 0) {
    if (!ws) return FP8GEMM_EINVAL;
    a.tail_workers = pl.tc.tail_workers;
    a.partials = reinterpret_cast<float*>(ws + pl.part_off);
    a.flags = reinterpret_cast<unsigned long long*>(ws + pl.flag_off);
    // a distinct, well-mixed value per call (the splitmix64 finaliser of a
    // counter), so that neither old flags nor leftover workspace bytes match it
    unsigned long long z = d.calls.fetch_add(1) + 1;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    a.epoch = z ^ (z >> 31);  // a bijection of z >= 1, hence never 0
  }
  // TMA descriptors are only meaningful on the TMA path (and need K >= 1);
  // the realigning producer reads x and w through plain pointers.
  CUtensorMap tmA, tmB;
  std::memset(&tmA, 0, sizeof(tmA));
  std::memset(&tmB, 0, sizeof(tmB));
  const bool use_tma = !pl.pub.realign && K > 0;
  cudaError_t e;
  if (pl.pub.path == FP8GEMM_PATH_MAIN) {
    // each CTA of a pair loads 128 rows of x and half of the tile's w rows
    const int b_rows = pl.tc.ctas == 2 ? pl.tc.bn / 2 : pl.tc.bn;
    // Pair tiles with four producers read each stage's two K blocks of an
    // operand as one 3-D box when K % 128 == 0: half the TMA copies (square
    // 44.8 -> 44.3 us, MLP 264.2 -> 262.9 us, 512 x 4096 x 4096 14.07 ->
    // 13.84 us; interleaved A/B runs)
    a.kbox = (use_tma && pl.tc.ctas == 2 && pl.tc.epi == 4 && K % 128 == 0) ? 1 : 0;
    if (use_tma && (a.kbox ? (encode_operand_kblocks(&tmA, xa, M, K, lxa, 128, 2) != FP8GEMM_OK ||
                              encode_operand_kblocks(&tmB, wa, w_rows, K, lwa, b_rows, 2) !=
                                  FP8GEMM_OK)
                           : (encode_operand(&tmA, xa, M, K, lxa, 128) != FP8GEMM_OK ||
                              encode_operand(&tmB, wa, w_rows, K, lwa, b_rows) != FP8GEMM_OK)))
      return FP8GEMM_ELAUNCH;
    if (pl.tc.ctas == 2) {
      CUtensorMap tmY;
      std::memset(&tmY, 0, sizeof(tmY));
      if (a.vec_store && encode_output(&tmY, y, M, N) != FP8GEMM_OK) return FP8GEMM_ELAUNCH;
      e = launch_tc2(tmA, tmB, tmY, a, pl.tc, s);
    } else {
      e = launch_tc(tmA, tmB, a, pl.tc, s);
    }
  } else {
    if (use_tma) {
      const bool wide = pl.dec.kbs > 1;
      if (wide ? (encode_operand_kblocks(&tmA, wa, N, K, lwa, 128, pl.dec.kbs) != FP8GEMM_OK ||
                  encode_operand_kblocks(&tmB, xa, M, K, lxa, pl.dec.mp, pl.dec.kbs) !=
                      FP8GEMM_OK)
               : (encode_operand(&tmA, wa, N, K, lwa, 128) != FP8GEMM_OK ||
                  encode_operand(&tmB, xa, M, K, lxa, pl.dec.mp) != FP8GEMM_OK))
        return FP8GEMM_ELAUNCH;
    }
    e = launch_decode(tmA, tmB, a, pl.dec, s);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ELAUNCH;
  }
  return FP8GEMM_OK;
}

}  // namespace

// Repitch workspace of fp8_gemm_scaled_noalloc, for callers that cannot
// allocate device memory.  In host code this name is only a stand-in: its
// device address comes from cudaGetSymbolAddress (noalloc_workspace below).
static __device__ __align__(256) unsigned char g_noalloc_workspace[FP8GEMM_NOALLOC_WORKSPACE_BYTES];

namespace {

// Device address of g_noalloc_workspace on device `dev`, which must be the
// current device; looked up on the first call on that device.
int noalloc_workspace(DevState& d, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!d.noalloc_ws) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return FP8GEMM_ELAUNCH;
    }
    d.noalloc_ws = p;
  }
  *out = static_cast<uint8_t*>(d.noalloc_ws);
  return FP8GEMM_OK;
}

// Enqueue a planned call whose workspace `ws` (pl.pub.workspace_bytes) is
// in hand: the repitch copies first, if any, then the GEMM on the operands it
// reads.
int run_with_workspace(const Plan& pl, DevState& d, const void* x, size_t ldx, const void* w,
                       size_t ldw, int K, const float* scale, void* y, int M, int N,
                       uint8_t* ws, cudaStream_t s) {
  if (!pl.pub.repitch) return launch_gemm(pl, d, x, ldx, w, ldw, K, scale, y, M, N, ws, s);
  RepitchArgs r{};
  r.x = static_cast<const uint8_t*>(x);
  r.w = static_cast<const uint8_t*>(w);
  r.xo = ws + pl.x_off;
  r.wo = ws + pl.w_off;
  r.K = K;
  r.Kp = pl.Kp;
  r.rows_x = pl.rx ? M : 0;
  r.rows_w = pl.rw ? N : 0;
  r.ldx = static_cast<long long>(ldx);
  r.ldw = static_cast<long long>(ldw);
  r.pdl = pdl_ok(s) ? 1 : 0;
  if (launch_repitch(r, s) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ELAUNCH;
  }
  return launch_gemm(pl, d, pl.rx ? static_cast<const void*>(r.xo) : x,
                     pl.rx ? static_cast<size_t>(pl.Kp) : ldx,
                     pl.rw ? static_cast<const void*>(r.wo) : w,
                     pl.rw ? static_cast<size_t>(pl.Kp) : ldw, K, scale, y, M, N, ws, s);
}

}  // namespace
}  // namespace fp8g

using namespace fp8g;

extern "C" int fp8_gemm_scaled_ex(const void* x, const void* w, const float* scale, void* y,
                                  int M, int N, int K, const fp8gemm_options* opt,
                                  fp8gemm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return FP8GEMM_EINVAL;
  if (M == 0 || N == 0) return FP8GEMM_OK;
  if (!scale || !y || (K > 0 && (!x || !w))) return FP8GEMM_EINVAL;
  if ((reinterpret_cast<uintptr_t>(scale) & 3u) || (reinterpret_cast<uintptr_t>(y) & 1u))
    return FP8GEMM_EALIGN;
  const size_t ldx = (opt && opt->ldx) ? opt->ldx : static_cast<size_t>(K);
  const size_t ldw = (opt && opt->ldw) ? opt->ldw : static_cast<size_t>(K);
  if (ldx < static_cast<size_t>(K) || ldw < static_cast<size_t>(K)) return FP8GEMM_EINVAL;
  // bytes spanned by each operand (the last row is K bytes long)
  const size_t xb = K > 0 ? (static_cast<size_t>(M) - 1) * ldx + static_cast<size_t>(K) : 0;
  const size_t wb = K > 0 ? (static_cast<size_t>(N) - 1) * ldw + static_cast<size_t>(K) : 0;
  const size_t yb = static_cast<size_t>(M) * static_cast<size_t>(N) * 2u;
  const size_t sb = static_cast<size_t>(N) * 4u;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || overlaps(y, yb, scale, sb))
    return FP8GEMM_EINVAL;
  const int dev = pointer_device(y);
  if (dev < 0 || pointer_device(scale) != dev ||
      (K > 0 && (pointer_device(x) != dev || pointer_device(w) != dev)))
    return FP8GEMM_EINVAL;
  const DeviceGuard guard(dev);
  if (!guard.ok()) return FP8GEMM_EDEVICE;
  DevState* d = nullptr;
  int st = device_state(dev, &d);
  if (st != FP8GEMM_OK) return st;
  Plan pl;
  st = make_plan(*d, x, w, M, N, K, opt, &pl);
  if (st != FP8GEMM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t need = pl.pub.workspace_bytes;
  if (need == 0) return launch_gemm(pl, *d, x, ldx, w, ldw, K, scale, y, M, N, nullptr, s);

  // workspace (repitch copies and/or split-tail partial sums): the caller's,
  // else the one the device keeps for this stream, else (while the stream is
  // being captured into a CUDA graph, whose replays may run on any stream,
  // or when the device keeps workspaces for too many other streams) one
  // taken for this call in stream order
  if (opt && opt->workspace) {
    uint8_t* ws = static_cast<uint8_t*>(opt->workspace);
    if (opt->workspace_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
        pointer_device(ws) != dev || overlaps(ws, need, y, yb) || overlaps(ws, need, x, xb) ||
        overlaps(ws, need, w, wb) || overlaps(ws, need, scale, sb))
      return FP8GEMM_EINVAL;
    return run_with_workspace(pl, *d, x, ldx, w, ldw, K, scale, y, M, N, ws, s);
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ELAUNCH;
  }
  if (cap == cudaStreamCaptureStatusNone) {
    unsigned long long sid = 0;
    if (cudaStreamGetId(s, &sid) != cudaSuccess) {
      cudaGetLastError();
      return FP8GEMM_ELAUNCH;
    }
    std::lock_guard<std::mutex> lk(d->ws_mu);
    uint8_t* ws = nullptr;
    st = stream_workspace(*d, dev, sid, need, s, &ws);
    if (st != FP8GEMM_OK) return st;
    if (ws) return run_with_workspace(pl, *d, x, ldx, w, ldw, K, scale, y, M, N, ws, s);
  }
  void* p = nullptr;
  const cudaError_t ae = cap == cudaStreamCaptureStatusNone
                             ? [&]() {
                                 cudaMemPool_t pool = workspace_pool(*d, dev);
                                 return pool ? cudaMallocFromPoolAsync(&p, need, pool, s)
                                             : cudaErrorMemoryAllocation;
                               }()
                             : cudaMallocAsync(&p, need, s);
  if (ae != cudaSuccess || !p) {
    cudaGetLastError();
    return FP8GEMM_ENOMEM;
  }
  st = run_with_workspace(pl, *d, x, ldx, w, ldw, K, scale, y, M, N, static_cast<uint8_t*>(p), s);
  if (cudaFreeAsync(p, s) != cudaSuccess) {
    cudaGetLastError();
    if (st == FP8GEMM_OK) st = FP8GEMM_ELAUNCH;
  }
  return st;
}

// Same layer as fp8_gemm_scaled for callers that must not allocate: the
// repitch copies (if any) go into the static g_noalloc_workspace instead of a
// pool or caller buffer.  Calls that overlap on the GPU race on that array.
extern "C" int fp8_gemm_scaled_noalloc(const void* x, const void* w, const float* scale, void* y,
                                       int M, int N, int K, fp8gemm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return FP8GEMM_EINVAL;
  if (M == 0 || N == 0) return FP8GEMM_OK;
  if (!scale || !y || (K > 0 && (!x || !w))) return FP8GEMM_EINVAL;
  if ((reinterpret_cast<uintptr_t>(scale) & 3u) || (reinterpret_cast<uintptr_t>(y) & 1u))
    return FP8GEMM_EALIGN;
  const size_t xb = static_cast<size_t>(M) * static_cast<size_t>(K);
  const size_t wb = static_cast<size_t>(N) * static_cast<size_t>(K);
  const size_t yb = static_cast<size_t>(M) * static_cast<size_t>(N) * 2u;
  const size_t sb = static_cast<size_t>(N) * 4u;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || overlaps(y, yb, scale, sb))
    return FP8GEMM_EINVAL;
  const int dev = pointer_device(y);
  if (dev < 0 || pointer_device(scale) != dev ||
      (K > 0 && (pointer_device(x) != dev || pointer_device(w) != dev)))
    return FP8GEMM_EINVAL;
  const DeviceGuard guard(dev);
  if (!guard.ok()) return FP8GEMM_EDEVICE;
  DevState* d = nullptr;
  int st = device_state(dev, &d);
  if (st != FP8GEMM_OK) return st;
  uint8_t* ws = nullptr;
  st = noalloc_workspace(*d, &ws);
  if (st != FP8GEMM_OK) return st;
  // plan as fp8_gemm_scaled would, with the static array as the workspace
  fp8gemm_options o;
  std::memset(&o, 0, sizeof(o));
  o.workspace = ws;
  o.workspace_bytes = FP8GEMM_NOALLOC_WORKSPACE_BYTES;
  Plan pl;
  st = make_plan(*d, x, w, M, N, K, &o, &pl);
  if (st != FP8GEMM_OK) return st;
  if (pl.pub.workspace_bytes > FP8GEMM_NOALLOC_WORKSPACE_BYTES) return FP8GEMM_ESIZE;
  return run_with_workspace(pl, *d, x, static_cast<size_t>(K), w, static_cast<size_t>(K), K,
                            scale, y, M, N, ws, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fp8_gemm_prepare_weight(const void* w, int N, int K, void* w_out,
                                       size_t ldw_out, fp8gemm_stream_t stream) {
  if (N < 0 || K < 0) return FP8GEMM_EINVAL;
  if (N == 0 || K == 0) return FP8GEMM_OK;
  if (!w || !w_out || ldw_out < static_cast<size_t>(K)) return FP8GEMM_EINVAL;
  if ((ldw_out % 16u) != 0 || (reinterpret_cast<uintptr_t>(w_out) & 15u)) return FP8GEMM_EALIGN;
  if (ldw_out > 0x7FFFFFFFu) return FP8GEMM_EINVAL;
  const size_t wb = static_cast<size_t>(N) * static_cast<size_t>(K);
  const size_t ob = (static_cast<size_t>(N) - 1) * ldw_out + ldw_out;
  if (overlaps(w, wb, w_out, ob)) return FP8GEMM_EINVAL;
  const int dev = pointer_device(w_out);
  if (dev < 0 || pointer_device(w) != dev) return FP8GEMM_EINVAL;
  const DeviceGuard guard(dev);
  if (!guard.ok()) return FP8GEMM_EDEVICE;
  DevState* d = nullptr;
  int st = device_state(dev, &d);
  if (st != FP8GEMM_OK) return st;
  RepitchArgs r{};
  r.w = static_cast<const uint8_t*>(w);
  r.wo = static_cast<uint8_t*>(w_out);
  r.K = K;
  r.Kp = static_cast<int>(ldw_out);
  r.rows_x = 0;
  r.rows_w = N;
  r.ldw = K;
  r.pdl = pdl_ok(reinterpret_cast<cudaStream_t>(stream)) ? 1 : 0;
  if (launch_repitch(r, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ELAUNCH;
  }
  return FP8GEMM_OK;
}

extern "C" int fp8_gemm_grouped(const void* x, const void* w, const float* scale, void* y,
                                const int* offsets, int groups, int M, int N, int K,
                                const fp8gemm_options* opt, fp8gemm_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || groups < 0) return FP8GEMM_EINVAL;
  if (M == 0 || N == 0 || groups == 0) return FP8GEMM_OK;
  if (K == 0 || !x || !w || !scale || !y || !offsets) return FP8GEMM_EINVAL;
  if (static_cast<long long>(groups) * N > 0x7FFFFFFFLL) return FP8GEMM_EINVAL;
  if ((reinterpret_cast<uintptr_t>(scale) & 3u) || (reinterpret_cast<uintptr_t>(y) & 1u) ||
      (reinterpret_cast<uintptr_t>(offsets) & 3u))
    return FP8GEMM_EALIGN;
  const size_t ldx = (opt && opt->ldx) ? opt->ldx : static_cast<size_t>(K);
  const size_t ldw = (opt && opt->ldw) ? opt->ldw : static_cast<size_t>(K);
  if (ldx < static_cast<size_t>(K) || ldw < static_cast<size_t>(K)) return FP8GEMM_EINVAL;
  const long long w_rows = static_cast<long long>(groups) * N;
  const size_t xb = (static_cast<size_t>(M) - 1) * ldx + static_cast<size_t>(K);
  const size_t wb = (static_cast<size_t>(w_rows) - 1) * ldw + static_cast<size_t>(K);
  const size_t yb = static_cast<size_t>(M) * static_cast<size_t>(N) * 2u;
  const size_t sb = static_cast<size_t>(w_rows) * 4u;
  const size_t ob = (static_cast<size_t>(groups) + 1u) * 4u;
  if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || overlaps(y, yb, scale, sb) ||
      overlaps(y, yb, offsets, ob))
    return FP8GEMM_EINVAL;
  const int dev = pointer_device(y);
  if (dev < 0 || pointer_device(scale) != dev || pointer_device(x) != dev ||
      pointer_device(w) != dev || pointer_device(offsets) != dev)
    return FP8GEMM_EINVAL;
  const DeviceGuard guard(dev);
  if (!guard.ok()) return FP8GEMM_EDEVICE;
  DevState* d = nullptr;
  int st = device_state(dev, &d);
  if (st != FP8GEMM_OK) return st;
  // CTA-pair tiles chosen as for one group of M rows; the work list (tiles of
  // every group) is built on the device, so every resident pair is launched.
  fp8gemm_options o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (o.path == FP8GEMM_PATH_DECODE || o.mma_ctas == 1 || o.force_realign) return FP8GEMM_EUNSUPPORTED;
  // the grouped layer reads its operands with TMA only
  if ((ldx % 16) || (ldw % 16) || !aligned16(x) || !aligned16(w)) return FP8GEMM_EALIGN;
  o.path = FP8GEMM_PATH_MAIN;
  o.mma_ctas = 2;
  o.split_tail = 0;
  o.no_workspace = 1;
  o.workspace = nullptr;
  o.workspace_bytes = 0;
  Plan pl;
  st = make_plan(*d, x, w, M, N, K, &o, &pl);
  if (st != FP8GEMM_OK) return st;
  if (pl.pub.realign || pl.pub.repitch) return FP8GEMM_EALIGN;
  const int pairs = tc2_pairs(*d, pl.tc.bn, pl.tc.stages, pl.tc.epi);
  if (pairs <= 0) return FP8GEMM_ELAUNCH;
  pl.tc.grid = 2 * pairs;
  pl.tc.tail_workers = 0;
  return launch_gemm(pl, *d, x, ldx, w, ldw, K, scale, y, M, N, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), offsets, groups);
}

extern "C" int fp8_gemm_scaled(const void* x, const void* w, const float* scale, void* y, int M,
                               int N, int K, fp8gemm_stream_t stream) {
  return fp8_gemm_scaled_ex(x, w, scale, y, M, N, K, nullptr, stream);
}

extern "C" int fp8_gemm_plan(int device, const void* x, const void* w, int M, int N, int K,
                             const fp8gemm_options* opt, fp8gemm_plan* out) {
  if (!out || M < 0 || N < 0 || K < 0) return FP8GEMM_EINVAL;
  if (device < 0 || device >= kMaxDevices) return FP8GEMM_EDEVICE;
  const DeviceGuard guard(device);
  if (!guard.ok()) return FP8GEMM_EDEVICE;
  DevState* d = nullptr;
  int st = device_state(device, &d);
  if (st != FP8GEMM_OK) return st;
  Plan pl;
  st = make_plan(*d, x, w, M, N, K, opt, &pl);
  if (st != FP8GEMM_OK) return st;
  *out = pl.pub;
  return FP8GEMM_OK;
}

extern "C" size_t fp8_gemm_workspace_bytes(int device, const void* x, const void* w, int M, int N,
                                           int K, const fp8gemm_options* opt) {
  fp8gemm_plan p;
  if (fp8_gemm_plan(device, x, w, M, N, K, opt, &p) != FP8GEMM_OK) return 0;
  return p.workspace_bytes;
}

extern "C" int fp8_gemm_check_device_error(fp8gemm_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_EDEVICE;
  }
  DevState* d = nullptr;
  int st = device_state(dev, &d);
  if (st != FP8GEMM_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ELAUNCH;
  }
  unsigned bits = 0;
  const unsigned zero = 0;
  if (cudaMemcpy(&bits, d->err_word, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(d->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_ELAUNCH;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_last_error_bits = bits;
  }
  return bits ? FP8GEMM_ETIMEOUT : FP8GEMM_OK;
}

extern "C" unsigned fp8_gemm_last_device_error_bits(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_last_error_bits;
}

extern "C" int fp8_gemm_set_wait_budget_ns(unsigned long long ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_budget_ns = ns ? ns : kDefaultBudgetNs;
  return FP8GEMM_OK;
}

extern "C" int fp8_gemm_selftest_wait_timeout(unsigned long long budget, fp8gemm_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FP8GEMM_EDEVICE;
  }
  DevState* d = nullptr;
  int st = device_state(dev, &d);
  if (st != FP8GEMM_OK) return st;
  if (budget == 0 || budget > 10000000000ull) return FP8GEMM_EINVAL;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(d->err_word, budget);
  if (cudaGetLastError() != cudaSuccess) return FP8GEMM_ELAUNCH;
  return FP8GEMM_OK;
}

extern "C" const char* fp8_gemm_status_string(int status) {
  switch (status) {
    case FP8GEMM_OK: return "ok";
    case FP8GEMM_EINVAL: return "invalid argument (null or host pointer, bad size, overlapping buffers)";
    case FP8GEMM_EALIGN: return "misaligned pointer (scale needs 4 bytes, y needs 2 bytes)";
    case FP8GEMM_EDEVICE: return "no usable device (needs compute capability 10.3)";
    case FP8GEMM_ELAUNCH: return "CUDA launch or runtime call failed";
    case FP8GEMM_ETIMEOUT: return "a kernel gave up a bounded wait; its output is invalid";
    case FP8GEMM_EUNSUPPORTED: return "requested configuration is not built";
    case FP8GEMM_ESIZE:
      return "fp8_gemm_scaled_noalloc: the repitch workspace this call needs exceeds "
             "FP8GEMM_NOALLOC_WORKSPACE_BYTES";
    case FP8GEMM_ENOMEM:
      return "no device memory for the workspace this call needs (pass one in "
             "fp8gemm_options.workspace, or set no_workspace)";
    default: return "unknown status";
  }
}

extern "C" int fp8_gemm_version(void) { return FP8GEMM_VERSION; }
