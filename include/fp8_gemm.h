/*
 * fp8_gemm.h -- C ABI of the GB300 (sm_103a) per-output-channel scaled FP8
 * linear layer.
 *
 *     y[m, n] = bf16_rn( (sum_k x[m, k] * w[n, k], accumulated in fp32)
 *                        * weight_scale[n] )
 *
 * The operation is the FP8 GEMM audited on the kernelbench.com model pages:
 * E4M3 operands with fp32 accumulation ("Kimi K3 (256k)" page, SM120 FP8 GEMM
 * paragraph; "deepseek-v4-flash" page, CUTLASS SM90 paragraph), the live
 * per-output-channel weight_scale applied to the accumulator in the epilogue
 * and a bf16 result ("Kimi K3 (256k)" page, SM90 WGMMA and sm_100 tcgen05
 * paragraphs; "claude-fable-5" page, CUTLASS 4.0 SM100 paragraph), over the
 * problem's large-M, M = 32 decode and K = 4127 shapes.
 *
 * Conventions shared by every entry point:
 *   - Status: every function returns an fp8gemm_status (0 = OK).  No
 *     exception or signal crosses the ABI.
 *   - Streams: `stream` is a CUDA runtime stream handle (cudaStream_t); NULL
 *     means the legacy default stream.  Compute calls are asynchronous with
 *     respect to the host and never synchronise.
 *   - Ownership: the caller owns every buffer.  The library keeps, per
 *     device, its properties, a 4-byte device error word (see
 *     fp8_gemm_check_device_error) and a few workspaces.  A call needs a
 *     workspace (see fp8_gemm_workspace_bytes) only for repitched copies of
 *     x and w whose rows TMA cannot tile, and for the optional split tail's
 *     partial sums.  It uses the caller's when fp8gemm_options.workspace is
 *     given.  Otherwise it uses the workspace the device keeps for the
 *     call's stream: taken from a private stream-ordered pool on that
 *     stream's first such call, enlarged in the stream's order when a call
 *     needs more, and kept until the process exits, so later calls on the
 *     stream allocate nothing; calls on one stream are ordered by the stream,
 *     so they never use it at the same time.  Streams are told apart by
 *     cudaStreamGetId.  Workspaces are kept for at most 16 streams per
 *     device; a call on a further stream, or on a stream being captured into
 *     a CUDA graph (whose replays may run on any stream), takes its workspace
 *     for itself in stream order (cudaMallocFromPoolAsync / cudaMallocAsync
 *     and cudaFreeAsync; a capture records these as graph memory nodes).  If
 *     the memory cannot be had the call returns FP8GEMM_ENOMEM and launches
 *     nothing.
 *   - Nothing derived from the data is ever cached: each call reads x, w
 *     and weight_scale as they are when the kernel runs (the pages' stale
 *     padded-input failure, "qwen3.8-max" page, odd-K pad-cache paragraph,
 *     is impossible by construction).
 *   - Thread safety: calls may come from several host threads.
 *   - Devices: a call works on the device that holds y (all buffers must be
 *     on it).  It makes that device current only while it runs and makes the
 *     caller's current device current again before it returns, on every
 *     return path; fp8_gemm_plan does the same for its `device` argument.
 *   - CUDA graphs: a call can be captured into a graph once the device has
 *     been set up by an earlier call; replays read the buffers as they are
 *     then.  A captured call that needs a workspace and brings none records
 *     its own allocation in the graph (see Ownership).  Consecutive
 *     calls on a stream are launched with programmatic stream serialization:
 *     each kernel may start its set-up while the previous one drains, and
 *     touches global memory only after it has completed.
 */
#ifndef FP8_GEMM_H
#define FP8_GEMM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA runtime stream handle without including CUDA headers
 * (identical to cudaStream_t). */
typedef struct CUstream_st *fp8gemm_stream_t;

#define FP8GEMM_VERSION 6

typedef enum {
    FP8GEMM_OK = 0,
    FP8GEMM_EINVAL = 1,    /* null pointer, bad size, host pointer, aliasing y */
    FP8GEMM_EALIGN = 2,    /* weight_scale not 4-byte or y not 2-byte aligned */
    FP8GEMM_EDEVICE = 3,   /* no CUDA device, or not compute capability 10.3 */
    FP8GEMM_ELAUNCH = 4,   /* the CUDA launch (or a CUDA runtime call) failed */
    FP8GEMM_ETIMEOUT = 5,  /* a kernel gave up a bounded wait (results invalid) */
    FP8GEMM_EUNSUPPORTED = 6, /* the options ask for a configuration not built */
    FP8GEMM_ESIZE = 7,     /* fp8_gemm_scaled_noalloc: workspace needed exceeds
                              FP8GEMM_NOALLOC_WORKSPACE_BYTES */
    FP8GEMM_ENOMEM = 8     /* no device memory for the workspace the call needs */
} fp8gemm_status;

/* Kernel path. */
enum {
    FP8GEMM_PATH_AUTO = 0,    /* M <= 64, or M <= 192 with N <= 8192: decode path,
                                 else main path */
    FP8GEMM_PATH_MAIN = 1,    /* persistent tcgen05 tile kernel */
    FP8GEMM_PATH_DECODE = 2   /* split-K swap-AB kernel; needs M <= 256 (M > 128
                                 only with 16-byte aligned rows or a workspace) */
};

/*
 * Optional tuning and test knobs; a zero-initialised struct (or NULL)
 * means "choose automatically".
 */
typedef struct {
    int path;           /* FP8GEMM_PATH_* */
    int force_realign;  /* 1: load operands with the in-kernel realigning
                           producer even when TMA could (tests that loader) */
    int tile_n;         /* main path N tile: 0 auto, or 128, 160, 192, 224, 256;
                           64 with one-CTA tiles only.  Decode path: 128-byte K
                           blocks per pipeline stage, 0 auto, 1, 2 or 4 (2 and 4
                           read each stage with one 3-D TMA box and need
                           K % 128 == 0 and rows TMA can read in place) */
    int stages;         /* pipeline depth: 0 auto */
    int splits;         /* decode path K splits (cluster size): 0 auto, 1..8 */
    int no_workspace;   /* 1: never repitch; rows TMA cannot tile are then
                           loaded by the in-kernel realigning producer */
    int mma_ctas;       /* main path: 0 auto, 1 one-CTA 128-row tiles,
                           2 CTA-pair 256-row tiles (tcgen05 cta_group::2) */
    int split_tail;     /* 1: share the last partial wave's tiles out by K
                           between CTA pairs (see fp8gemm_plan.split_tiles);
                           needs a workspace.  Off by default: with this
                           kernel's epilogue the fix-up costs about what it
                           saves */
    int reserved;       /* must be zero */
    void *workspace;    /* optional caller workspace (device, 256-byte aligned) */
    size_t workspace_bytes; /* its size; must be >= fp8_gemm_workspace_bytes() */
    size_t ldx;         /* row pitch of x in bytes (0 = K): row m starts at x + m * ldx;
                           the caller guarantees [x, x + (M-1)*ldx + K) is device memory */
    size_t ldw;         /* row pitch of w in bytes (0 = K).  An operand whose pitch is a
                           multiple of 16 and whose base is 16-byte aligned is read in
                           place by TMA whatever K is (bytes past K in a row are never
                           read); any other operand is repitched into the workspace
                           (or, with pitch == K, loaded by the realigning producer) */
    int epilogue_warps; /* CTA-pair tiles: 0 auto (8 when K <= 1024, every pair
                           has at least two tiles and there is no split tail,
                           else 4), 4, or 8 (K <= 3072, no split tail) */
} fp8gemm_options;

/* What a call with the same arguments would launch (see fp8_gemm_plan). */
typedef struct {
    int path;           /* FP8GEMM_PATH_MAIN or FP8GEMM_PATH_DECODE; 0 = no launch */
    int realign;        /* 1: operands loaded by the realigning producer */
    int tile_m;         /* rows of x per tile (main: 128, or 256 on a CTA pair) /
                           rows of w per tile (decode) */
    int tile_n;         /* columns of y per tile (main) / padded M (decode) */
    int stages;         /* shared-memory pipeline depth */
    int splits;         /* K splits (decode), 1 for main */
    int grid;           /* CTAs launched */
    int cluster;        /* CTAs per cluster (2 for CTA-pair tiles, splits for decode) */
    int threads;        /* threads per CTA */
    int smem_bytes;     /* dynamic shared memory per CTA */
    int launches;       /* kernels launched by one call (0, 1, or 2 with repitch) */
    int repitch;        /* 1: operands are first copied to a 64-byte pitch */
    int occupancy;      /* resident CTAs per SM of the GEMM kernel */
    int split_tiles;    /* main path, CTA pairs: tiles past the last full wave
                           whose K blocks are shared out between
                           tail_workers pairs (0 = no split) */
    int tail_workers;   /* CTA pairs sharing them; each publishes at most one
                           fp32 partial sum that the tile's owner adds */
    size_t workspace_bytes; /* device workspace the call needs (0 = none) */
    int epilogue_warps; /* warps scaling and storing y per CTA (4 or 8) */
    int kblocks_per_stage; /* 128-byte K blocks per pipeline stage (decode: 1, 2 or
                              4; main path: 2 on CTA pairs, 1 on one CTA) */
} fp8gemm_plan;

/*
 * fp8_gemm_scaled -- y = bf16((x . w^T, fp32 acc) * weight_scale), on `stream`.
 *
 *   x      device, E4M3FN bytes, [M, K] row-major (K contiguous), any alignment
 *   w      device, E4M3FN bytes, [N, K] row-major (nn.Linear layout), any alignment
 *   scale  device, fp32 [N], 4-byte aligned
 *   y      device, bf16 [M, N] row-major, 2-byte aligned; written, never read.
 *          Must not overlap x, w or scale.
 *   M,N,K  >= 0.  M == 0 or N == 0: nothing is launched.  K == 0: y = 0.
 *
 * Rows whose pitch K is not a multiple of 16 bytes (e.g. K = 4127), or
 * operands not 16-byte aligned, cannot be tiled by TMA.  They are first
 * copied by a repitch kernel into the workspace with a 64-byte pitch and zero
 * pad bytes (two launches); with no_workspace an in-kernel realigning
 * producer loads them directly instead (one launch, no workspace, but about
 * ten times slower on large shapes: its loads pass through registers).
 * Either way bytes past K count as zeros, which adds exactly nothing (the
 * zero-padding argument of the "Kimi K3 (256k)" page, SM100 Triton
 * paragraph).  No operand data is kept between calls.
 *
 * With fp8gemm_options.split_tail on CTA-pair tiles, when the tiles do not
 * fill the last wave of the persistent grid, that wave's tiles are cut along
 * K into two or three segments run by different CTA pairs
 * (fp8gemm_plan.split_tiles).  Every pair then ends after about the same
 * number of K blocks.  The pair that holds a tile's first K block adds the
 * other segment's fp32 partial sum (published through the workspace) to its
 * accumulator, then scales and rounds once, so results do not depend on
 * timing.  Without a workspace the last wave runs unsplit.
 *
 * Returns FP8GEMM_OK once the kernel is enqueued.  Errors inside the kernel
 * (a bounded wait that ran out) are reported by fp8_gemm_check_device_error.
 */
int fp8_gemm_scaled(const void *x, const void *w, const float *scale, void *y,
                    int M, int N, int K, fp8gemm_stream_t stream);

/* As fp8_gemm_scaled, with options (NULL = automatic). */
int fp8_gemm_scaled_ex(const void *x, const void *w, const float *scale, void *y,
                       int M, int N, int K, const fp8gemm_options *opt,
                       fp8gemm_stream_t stream);

/*
 * fp8_gemm_plan -- fill *out with what fp8_gemm_scaled_ex would launch for
 * these sizes on CUDA device `device`, without launching anything.  x and w
 * are used only for their alignment and may be NULL (taken as 16-byte
 * aligned).
 */
int fp8_gemm_plan(int device, const void *x, const void *w, int M, int N, int K,
                  const fp8gemm_options *opt, fp8gemm_plan *out);

/*
 * fp8_gemm_workspace_bytes -- device workspace (bytes) a call with these
 * arguments needs for its repitch pass and split tail; 0 when it needs none.  x and w are
 * used only for their alignment and may be NULL (taken as 16-byte aligned).
 * Returns 0 also for invalid arguments.
 */
size_t fp8_gemm_workspace_bytes(int device, const void *x, const void *w, int M, int N,
                                int K, const fp8gemm_options *opt);

/*
 * fp8_gemm_scaled_noalloc -- the same layer as fp8_gemm_scaled, for callers
 * that must not allocate device memory: code that runs where cudaMalloc is
 * forbidden or unsafe (inside another allocator's or framework's memory
 * accounting, in a context whose memory is fixed up front, on a path that
 * may not synchronise the device).  It calls no cudaMalloc, cudaFree, pool
 * or other allocating routine.  The pages have no counterpart; it is an
 * addition of this library.
 *
 * When the main path has to repitch x and w (rows not 16-byte aligned, e.g.
 * K = 4127), the copies go into one static device array of
 * FP8GEMM_NOALLOC_WORKSPACE_BYTES (32 MiB) that every GPU which loads the
 * library holds until the process exits.  The repitch kernel writes every
 * byte of it that the GEMM then reads, pad bytes included, so nothing has to
 * start at zero.  Calls that need more than that (M * Kp + N * Kp bytes,
 * Kp = round_up(K, 64), each part rounded up to 256 bytes) return
 * FP8GEMM_ESIZE and launch nothing.
 *
 * All calls on a device share the one array and it keeps the last call's
 * contents: two calls that overlap on the GPU (different streams with no
 * ordering between them) race on it and may produce wrong results.  Order
 * them on one stream, or with events.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current), which may load the
 * library's module; make that first call before any stream capture.
 * Arguments and layouts are those of fp8_gemm_scaled, and so is the error
 * behaviour, with two differences: a call whose workspace would exceed the
 * array returns FP8GEMM_ESIZE (it never switches to the slow in-kernel
 * loader on its own), and FP8GEMM_ENOMEM cannot occur.
 */
#define FP8GEMM_NOALLOC_WORKSPACE_BYTES (32u * 1024u * 1024u)
int fp8_gemm_scaled_noalloc(const void *x, const void *w, const float *scale, void *y,
                            int M, int N, int K, fp8gemm_stream_t stream);

/*
 * fp8_gemm_grouped -- the layer for `groups` independent weight groups (the
 * experts of a mixture-of-experts layer) in one launch:
 *
 *     y[m, n] = bf16_rn( (sum_k x[m, k] * w[g, n, k]) * weight_scale[g, n] )
 *               for every row m of group g
 *
 *   x        device, E4M3 [M, K] row-major: all groups' rows, group g's contiguous
 *   w        device, E4M3 [groups, N, K] row-major (group g's weight at row g * N)
 *   scale    device, fp32 [groups, N], 4-byte aligned
 *   y        device, bf16 [M, N] row-major; rows outside every group are not written
 *   offsets  device, int32 [groups + 1], 4-byte aligned: group g owns rows
 *            [offsets[g], offsets[g+1]).  Read by the kernel when it runs, so a
 *            routing kernel earlier on the stream may write them (no host
 *            synchronisation).  Values are clamped to [0, M] and made
 *            non-decreasing (a group starts no earlier than the previous one
 *            ends), so no two groups share a row whatever the table holds.
 *   M, N, K  K >= 1; groups * N < 2^31.
 *
 * The pages run grouped (MoE up-projection) GEMMs over expert offsets in
 * bf16 ("Kimi K3 (256k)", "qwen3.8-max" and "claude-fable-5" pages, MoE
 * up-projection paragraphs); here the CTA-pair kernel walks every group's
 * 256-row tiles in one persistent work list built from the offsets on the
 * device.  Operands must be readable by TMA in place: K (or the pitches
 * fp8gemm_options.ldx / ldw) a multiple of 16 and 16-byte aligned bases, else
 * FP8GEMM_EALIGN.  Options that select the decode path, one-CTA tiles or the
 * realigning loader return FP8GEMM_EUNSUPPORTED; tile_n and stages apply.
 */
int fp8_gemm_grouped(const void *x, const void *w, const float *scale, void *y,
                     const int *offsets, int groups, int M, int N, int K,
                     const fp8gemm_options *opt, fp8gemm_stream_t stream);

/*
 * fp8_gemm_prepare_weight -- copy w [N, K] (row pitch K, any alignment) to
 * w_out with row pitch ldw_out (a multiple of 16, >= K; w_out 16-byte
 * aligned), bytes [K, ldw_out) of each row set to zero.  Passing w_out with
 * fp8gemm_options.ldw = ldw_out then lets every later call read the weight
 * with TMA in place, so that only x is repitched per call when K % 16 != 0
 * (the pages cache a padded weight per weight version: "glm-5.2" page,
 * Triton TMA paragraph; "Kimi K3 (256k)" page, sm_100 tcgen05 paragraph;
 * here the caller owns the copy and decides when it is stale, and the
 * default path keeps nothing between calls).  A pitch that is a multiple of
 * 64 bytes is the fast choice: rows an odd multiple of 16 bytes apart start
 * every 128-byte K block in the middle of a 32-byte sector, which slows the
 * GEMM by up to a sixth.  Asynchronous on `stream`; w_out must not overlap w.
 */
int fp8_gemm_prepare_weight(const void *w, int N, int K, void *w_out, size_t ldw_out,
                            fp8gemm_stream_t stream);

/*
 * fp8_gemm_check_device_error -- synchronise `stream`, read and clear the
 * device error word of the current device.  FP8GEMM_ETIMEOUT means some
 * kernel launched since the last check gave up a bounded wait and its output
 * is invalid; FP8GEMM_ELAUNCH means the stream reported a CUDA error.
 */
int fp8_gemm_check_device_error(fp8gemm_stream_t stream);

/* Raw value of the device error word as last read by
 * fp8_gemm_check_device_error (bit flags; 0 = none). */
unsigned fp8_gemm_last_device_error_bits(void);

/* Longest single wait inside a kernel, in nanoseconds (default 1e9, or the
 * FP8GEMM_WAIT_BUDGET_NS environment variable at load).  0 restores the
 * default.  Applies to launches made after the call. */
int fp8_gemm_set_wait_budget_ns(unsigned long long ns);

/*
 * fp8_gemm_selftest_wait_timeout -- launch one tiny kernel whose single
 * thread waits on an mbarrier that nothing ever completes, with the given
 * budget (ns).  The wait must run out, record its error bit and return, so
 * that fp8_gemm_check_device_error then reports FP8GEMM_ETIMEOUT and the
 * context stays usable.  Exercises the bounded-wait machinery every kernel
 * relies on, without faulting or hanging the GPU.
 */
int fp8_gemm_selftest_wait_timeout(unsigned long long budget_ns, fp8gemm_stream_t stream);

/* Static description of a status code. */
const char *fp8_gemm_status_string(int status);

/* FP8GEMM_VERSION of the built library. */
int fp8_gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8_GEMM_H */
