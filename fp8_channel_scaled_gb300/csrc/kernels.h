// kernels.h -- internal interface between the C-ABI host code (api.cu) and
// the kernel translation units.  Not part of the public API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fp8g {

// Operands and bookkeeping shared by every GEMM kernel.
struct GemmArgs {
  const uint8_t* x;      // E4M3 [M, K] row-major
  const uint8_t* w;      // E4M3 [N, K] row-major
  const float* scale;    // fp32 [N]
  uint16_t* y;           // bf16 [M, N] row-major
  int M, N, K;
  int num_kb;            // ceil(K / 128)
  int vec_store;         // 1: y rows are 16-byte aligned (N % 8 == 0, y aligned)
  unsigned* err;         // device error word
  unsigned long long budget_ns;  // longest single wait before giving up
  // Split tail of the CTA-pair kernel (tail_workers == 0: no split; see
  // WorkIter in sched.cuh): slot q < tail_workers of `partials` holds worker
  // q's published partial sum, [2 CTAs][4 warps][BN / 32 chunks][32 columns]
  // [32 rows] fp32; flags[q][2][4] is set to `epoch` once the matching
  // warp's part is written.  Epochs are unique per device and call, so the
  // flags never need clearing.
  int tail_workers;
  float* partials;
  unsigned long long* flags;
  unsigned long long epoch;
  // Grouped layer (CTA-pair kernel only; group_offsets == nullptr: one
  // group): rows [offs[g], offs[g+1]) of x and y belong to group g, whose
  // weight is rows [g N, (g+1) N) of w and whose scales are scale[g N ..].
  // The offsets are read on the device; values outside [0, M] are clamped.
  const int* group_offsets;  // device, groups + 1 entries
  int groups;
  int pdl;  // host side: launch with programmatic stream serialization
  // CTA-pair kernel with four producer warps: 1 when each stage's two K
  // blocks of an operand are one 3-D box (tensor maps [K / 128][rows][128
  // bytes], K % 128 == 0), 0 when each K block is its own 2-D box
  int kbox;
};

// ---- persistent tcgen05 kernel (large M) ---------------------------------
struct TcConfig {
  int ctas;        // 1: one-CTA 128-row tiles; 2: CTA-pair 256-row tiles (gemm_tc2.cu)
  int bn;          // N tile; the K block is 128 bytes
  int stages;      // shared-memory pipeline depth
  bool realign;    // operands loaded by the realigning producer instead of TMA
  int grid;        // persistent CTAs
  int group_m;     // M tiles per raster group
  int tail_workers;  // CTA pairs sharing the split tail (0: no split; pair kernel only)
  int epi;         // pair kernel: epilogue warps, 4 or 8 (8: short-K tiles, no split tail)
};
bool tc_config_supported(int bn, int stages, bool realign);
int tc_smem_bytes(int bn, int stages, bool realign);
int tc_threads(bool realign);
int tc_max_stages(int bn, bool realign, int smem_optin);
cudaError_t tc_prepare(int bn, int stages, bool realign);  // per device, before first launch
cudaError_t tc_blocks_per_sm(int bn, int stages, bool realign, int* out);
cudaError_t launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                      const TcConfig& c, cudaStream_t s);

// ---- persistent tcgen05 kernel on CTA pairs (large M) -----------------------
bool tc2_config_supported(int bn, int stages, int epi);
int tc2_smem_bytes(int bn, int stages, int epi);
int tc2_threads(int epi);
int tc2_max_stages(int bn, int smem_optin, int epi);
cudaError_t tc2_prepare(int bn, int stages, int epi);
cudaError_t tc2_max_active_pairs(int bn, int stages, int epi, int grid, int* out);
cudaError_t launch_tc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                       const GemmArgs& a, const TcConfig& c, cudaStream_t s);

// ---- split-K decode kernel (small M, swap-AB, cluster reduce) -------------
// Programmatic dependent launch: the kernel may be launched, and run its
// prologue, while the previous kernel of the stream is still finishing.  Each
// kernel of this library waits in griddep_wait() before it touches global
// memory, so stream order still holds for every byte it reads or writes.
// Launches use it only when the host allows it for the stream (see pdl_ok in
// api.cu): during stream capture a programmatic edge can only leave a kernel.
inline void set_pdl(cudaLaunchAttribute& attr) {
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
}

struct DecConfig {
  int mp;          // M padded to the MMA N dimension (32, 64 or 128)
  int stages;      // shared-memory pipeline depth
  bool realign;    // operands loaded by the realigning producer instead of TMA
  int splits;      // K splits = cluster size (1..8)
  int n_tiles;     // ceil(N / 128)
  int kbs;         // 128-byte K blocks per stage (> 1: 3-D tensor maps, K % 128 == 0)
};
bool dec_config_supported(int mp, int stages, bool realign, int kbs);
int dec_smem_bytes(int mp, int stages, bool realign, int kbs);
int dec_threads(bool realign);
int dec_tmem_cols(int mp);
int dec_stage_bytes(int mp, int kbs);  // shared-memory bytes of one ring stage (TMA path)
cudaError_t dec_prepare(int mp, int stages, bool realign, int kbs);
cudaError_t dec_blocks_per_sm(int mp, int stages, bool realign, int kbs, int* out);
cudaError_t dec_max_active_clusters(int mp, int stages, bool realign, int kbs, int splits,
                                    int grid, int* out);
cudaError_t launch_decode(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                          const DecConfig& c, cudaStream_t s);


// ---- repitch of unaligned operands into a workspace ------------------------
struct RepitchArgs {
  const uint8_t* x;      // [rows_x, K] with row pitch ldx bytes, any alignment
  const uint8_t* w;      // [rows_w, K] with row pitch ldw bytes, any alignment
  uint8_t* xo;           // [rows_x, Kp], 16-byte aligned
  uint8_t* wo;           // [rows_w, Kp], 16-byte aligned
  int K, Kp;             // Kp = a multiple of 16 >= K; bytes [K, Kp) of each row are set to 0
  long long rows_x;      // M, or 0 to leave x alone
  long long rows_w;      // N, or 0 to leave w alone
  long long ldx, ldw;    // source row pitches (>= K)
  int pdl;               // launch with programmatic stream serialization
};
cudaError_t launch_repitch(const RepitchArgs& a, cudaStream_t s);

}  // namespace fp8g
