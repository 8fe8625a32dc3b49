/*
 * w4.h -- C ABI of libw4: fused 4-bit weight-only dequant-GEMV (W4A16) for GB300 (sm_103a).
 *
 * Formats
 *   NF4  ("LLM Quantization on RTX 4060: Where 4-bit Decode Falls Behind FP16",
 *         section "Standard Expectation from Quantization"): a 16-entry normal-float code
 *         book, blocks of `blocksize` (default 64) consecutive weights of one row share one
 *         FP32 absmax, two 4-bit codes per byte.
 *   INT4 ("My Triton Kernel Ties bitsandbytes -- and Both Lose to Math", section "The kernels":
 *         the +8 zero point; group size 128 as in "LLM Compressor 0.14: GPTQ's 15x speedup is
 *         one fused loop", section "How the 15x and 30x were measured"): groups of `group`
 *         weights of one row share one FP16 scale = absmax / 7; the nibble holds q + 8.
 *   FP4  (E2M1: "LLM Compressor 0.14: GPTQ's 15x speedup is one fused loop", section "Details
 *         worth knowing": the grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} and its threshold ladder, ties
 *         to the even code): groups of `group` (default 32) weights of one row share one FP16
 *         scale = absmax / 6; the nibble holds the sign in bit 3 and the grid index in bits 0-2.
 *
 * Layouts (row-major, "out x in" = N x K, as the fused kernel of the first page indexes them,
 * section "Kernel Implementation")
 *   packed  uint8  [N][K/2]   byte j of a row = (code of element 2j) << 4 | code of element 2j+1
 *   absmax  float  [N][K/blocksize]            (NF4)
 *   scale   fp16   [N][K/group]                (INT4, FP4; IEEE binary16 bits in uint16_t)
 *   codebook float [16], ascending             (NF4)
 *   x       fp16   [M][K]   activations, M = batch (1 ... 128)
 *   y       fp16   [M][N]   y[m][n] = sum_k w_hat[n][k] * x[m][k], accumulated in FP32
 *
 * Ownership and execution
 *   Every pointer is a device pointer owned by the caller (except w4_nf4_codebook's output and
 *   the descriptor array of w4_gemv_sequence / w4_step_create, which are host memory).  No call
 *   allocates device memory on its launch path, none synchronises the device, and every launch
 *   goes to the given stream (NULL = legacy default stream).  y is overwritten completely: no
 *   pre-zeroing, no accumulation into y, repeated calls give identical bits.
 *
 *   GEMV kernels use programmatic dependent launch: a GEMV may start while the kernel before it
 *   in the stream is finishing, and it reads packed weights, scales and the code book before that
 *   kernel has completed; it reads x and writes y only after.  So weights, scales and code book
 *   must not be produced by the kernel that immediately precedes the GEMV in the same stream if
 *   that kernel signals early launch (only libw4's own GEMV kernels do, and they write only y).
 *
 * Errors
 *   Every call validates its arguments on the host before touching CUDA and returns a w4_status.
 *   W4_ERR_CUDA means a CUDA runtime call failed; w4_last_cuda_error() returns its cudaError_t.
 *   Device-side waits are bounded; a wait that runs out sets a device error word that
 *   w4_device_check() reads (it synchronises the stream) and reports as W4_ERR_TIMEOUT.
 */
#ifndef W4_H
#define W4_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t (struct CUstream_st*); declared here so that the header needs
 * no CUDA include. */
typedef struct CUstream_st* w4_stream_t;

typedef enum {
  W4_OK = 0,
  W4_ERR_NULL = -1,        /* a required pointer is NULL                                   */
  W4_ERR_SHAPE = -2,       /* M, N or K out of range; K not a multiple of the block size    */
  W4_ERR_ALIGN = -3,       /* a device pointer breaks the alignment its call states          */
  W4_ERR_BLOCKSIZE = -4,   /* block / group size is not a power of two in [32, 256]          */
  W4_ERR_CUDA = -5,        /* a CUDA runtime call failed; see w4_last_cuda_error()          */
  W4_ERR_TIMEOUT = -6,     /* a bounded device-side wait ran out (reported by w4_device_check) */
  W4_ERR_UNSUPPORTED = -7, /* valid arguments outside what this build implements           */
  W4_ERR_LIMIT = -8        /* beyond the fixed size of w4_gemv_levels_noalloc's counter array */
} w4_status;

typedef enum { W4_FMT_NF4 = 0, W4_FMT_INT4 = 1, W4_FMT_FP4 = 2 } w4_format;

/* Limits of this build. */
#define W4_MAX_BATCH 4096       /* M; above 128, batch tiles of 128 or 256 rows (prefill-sized) */
#define W4_MAX_K 10240          /* K; sizes the batch 1 ... 8 kernel's partial-sum buffers     */

/* ---------------------------------------------------------------------------------------
 * w4_nf4_codebook -- the 16 NF4 code values, ascending, FP32 (host function, no CUDA).
 * The pages name the standard NF4 code book without printing it; this is the QLoRA
 * construction ("4-bit NormalFloat", Dettmers et al. 2023): normal quantiles at
 * probabilities evenly spaced from delta = ((1 - 1/32) + (1 - 1/30)) / 2 down to 1/2, eight
 * on the positive side and seven on the negative side, an exact zero, all divided by the
 * largest; float64 arithmetic, one rounding to FP32.  Result: out[0] = -1, out[7] = 0,
 * out[15] = 1.  Returns W4_ERR_NULL if out is NULL.
 */
int w4_nf4_codebook(float out[16]);

/* ---------------------------------------------------------------------------------------
 * w4_quantize_nf4 -- block-wise NF4 quantisation of an FP32 matrix W [N][K] (device).
 * Per block of `blocksize` weights of a row: a = max |w| -> absmax; n = w / a (IEEE FP32
 * division; a == 0 gives n = 0); code = the nearest code-book value to n, a tie going to the
 * lower code (decided exactly: n is compared with the midpoints (c[i] + c[i+1]) / 2 in
 * float64); two codes per byte, element 2j in the high nibble ("LLM Quantization on RTX 4060",
 * sections "Standard Expectation from Quantization" and "Kernel Implementation").
 * codebook must be ascending.  W entries must be finite.
 * Sizes: N >= 1, blocksize <= K <= W4_MAX_K, K % blocksize == 0, blocksize a power of two in
 * [32, 256].  W, packed, absmax 16-byte aligned.  The same size rules hold for every call below.
 */
int w4_quantize_nf4(const float* W, uint8_t* packed, float* absmax, const float* codebook,
                    int N, int K, int blocksize, w4_stream_t stream);

/* w4_quantize_int4 -- group-wise INT4 with the +8 zero point ("My Triton Kernel Ties
 * bitsandbytes", section "The kernels").  Per group: s = fp16(absmax / 7) (the FP32 quotient
 * rounded to FP16); q = clamp(rint(w / s), -8, 7) + 8 with w / s an IEEE FP32 division and
 * rint rounding halves to even ("LLM Compressor 0.14", section "Details worth knowing");
 * s == 0 gives q = 8.  |w| must stay below 7 * 65504 (so that s is finite). */
int w4_quantize_int4(const float* W, uint8_t* packed, uint16_t* scale,
                     int N, int K, int group, w4_stream_t stream);

/* w4_quantize_fp4 -- group-wise FP4 (E2M1) with an FP16 scale ("LLM Compressor 0.14",
 * section "Details worth knowing").  Per group: s = fp16(absmax / 6) (the FP32 quotient rounded
 * to FP16); r = w / s (IEEE FP32 division); the grid index of |r| is found by a ladder over the
 * midpoints t of consecutive grid values, moving up past an even rung when |r| > t and past an
 * odd rung when |r| >= t, so that a value on a midpoint goes to the even index; |r| above 6
 * stays at index 7; code = (w < 0) << 3 | index.  s == 0 gives code 0 for the whole group.
 * |w| must stay below 6 * 65504. */
int w4_quantize_fp4(const float* W, uint8_t* packed, uint16_t* scale,
                    int N, int K, int group, w4_stream_t stream);

/* w4_dequantize_nf4 -- W_out[n][k] = code[q] * absmax (FP32 product), a test and
 * debugging aid; the GEMVs never materialise this matrix.  W_out 8-byte aligned. */
int w4_dequantize_nf4(const uint8_t* packed, const float* absmax, const float* codebook,
                      float* W_out, int N, int K, int blocksize, w4_stream_t stream);

/* w4_dequantize_int4 -- W_out[n][k] = (q - 8) * s, exact in FP32. */
int w4_dequantize_int4(const uint8_t* packed, const uint16_t* scale, float* W_out,
                       int N, int K, int group, w4_stream_t stream);

/* w4_dequantize_fp4 -- W_out[n][k] = (-1)^(bit 3) * grid[q & 7] * s, exact in FP32. */
int w4_dequantize_fp4(const uint8_t* packed, const uint16_t* scale, float* W_out,
                      int N, int K, int group, w4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * w4_gemv_nf4 / w4_gemv_int4 / w4_gemv_fp4 -- y = x . dequant(W)^T in one pass: packed weights
 * and scales
 * are streamed once, unpacked and decoded on chip and accumulated in FP32 against x; no
 * dequantised weight matrix is ever written ("LLM Quantization on RTX 4060", sections
 * "Fused Kernel: Moving Dequantization On-Chip" and "Kernel Implementation"; FP32
 * accumulation as that kernel's comment requires).  y is rounded to FP16 (nearest even).
 * Batches 1 ... 8 run in the persistent small-batch kernel (weights decoded through a byte-pair
 * table into warp-level mma.sync FP16 x FP16 -> FP32 products, block scales applied to the FP32
 * partial sums); batches 9 ... 128 on the 5th-generation tensor cores (tcgen05) when K is a
 * multiple of 64, else in 8-row launches of the small-batch kernel.  Larger batches
 * (prefill-sized, up to W4_MAX_BATCH) run as tiles of batch rows, each tile one pass over the
 * weights: 256 rows (one 256-column accumulator) where the matrix has at least half as many
 * 128-row tiles as the GPU has SMs, else 128.
 * Sizes: 1 <= M <= W4_MAX_BATCH, N >= 1, 32 <= K <= W4_MAX_K, K % blocksize == 0,
 * blocksize a power of two in [32, 256].  packed, scales, x 16-byte aligned; y 2-byte aligned.
 * Agreement with the float64 definition: relative L2 error <= 1e-3 and
 * max |error| <= 2e-2 * RMS(y) per output vector, under these conditions:
 *   all paths: every |x| <= 65504 (FP16 inputs) and |y| within the FP16 range;
 *   batches 1 ... 8: no condition on the scales (NF4 code values rounded to FP16, INT4 and FP4
 *     values exact in FP16; the FP32 / FP16 block scale multiplies the FP32 partial sum);
 *   batches 9 ... 128 (tcgen05, and the mma.sync fallback): each decoded weight is formed in
 *     FP16 as fp16(value) * fp16(scale), so an NF4 absmax must lie in [6.1e-5, 65504] (the FP16
 *     normal range; below it the rounded scale keeps fewer than 11 significant bits) and every
 *     decoded weight must stay below 65504; INT4 and FP4 scales are FP16 already.
 */
int w4_gemv_nf4(const uint8_t* packed, const float* absmax, const float* codebook,
                const uint16_t* x, uint16_t* y, int M, int N, int K, int blocksize,
                w4_stream_t stream);
int w4_gemv_int4(const uint8_t* packed, const uint16_t* scale,
                 const uint16_t* x, uint16_t* y, int M, int N, int K, int group,
                 w4_stream_t stream);
int w4_gemv_fp4(const uint8_t* packed, const uint16_t* scale,
                const uint16_t* x, uint16_t* y, int M, int N, int K, int group,
                w4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * w4_gemv_plan -- which kernel w4_gemv_nf4 / _int4 / _fp4 would run for these sizes, and its
 * launch geometry, on a GPU with sm_count SMs (152 on GB300).  The batch-driven choice of
 * path is the one "Do Quantization and Sparsity make LLM Inference Faster ?" describes for
 * bitsandbytes (section "NF4: fast at batch 1, slower at larger batches").  Host only: no
 * device call, nothing allocated; *plan is caller-owned and fully written on W4_OK.
 *   kernel      W4_KERNEL_SMALL_BATCH or W4_KERNEL_TCGEN05
 *   launches    kernel launches the call makes (small-batch kernel: one per <= batch_tile rows;
 *               batches above 128: one set per 128-row batch tile)
 *   batch_tile  batch rows per launch (small-batch kernel) or MMA N columns (tcgen05: 16/32/64/128)
 *   threads     threads per CTA; smem_bytes: dynamic shared memory per CTA
 *   stages      ring stages (small-batch kernel: packed tiles; tcgen05: x / A stages)
 *   grid        CTAs per launch (tcgen05), or 0 where the launch sizes it from occupancy
 *   cluster     CTAs per thread-block cluster splitting K (1: no split)
 * The figures are those of the widest launch.  The mma.sync tensor-core
 * kernel, which serves only if the driver cannot encode TMA descriptors, is not predicted.
 * Errors: W4_ERR_NULL (plan NULL), W4_ERR_UNSUPPORTED (format, M > W4_MAX_BATCH or a shape
 * no kernel takes), W4_ERR_SHAPE / W4_ERR_BLOCKSIZE as for the GEMV, W4_ERR_SHAPE for
 * sm_count < 1.
 */
typedef enum { W4_KERNEL_SMALL_BATCH = 1, W4_KERNEL_TCGEN05 = 2 } w4_kernel;
typedef struct {
  int kernel, launches, batch_tile, threads, smem_bytes, stages, grid, cluster;
} w4_gemv_plan_t;
int w4_gemv_plan(int format, int M, int N, int K, int blocksize, int sm_count, w4_gemv_plan_t* plan);

/* ---------------------------------------------------------------------------------------
 * Decode step: the projections of one decode step ("Do Quantization and Sparsity make LLM
 * Inference Faster ?", section "What we did": 197 GEMVs per token).  Descriptors carry a level:
 * levels start at 0 and never decrease along the array; the GEMVs of one level are independent
 * of each other (e.g. q, k and v, which read the same activation), and a level reads x only after
 * every GEMV of the earlier levels is complete.
 */
typedef struct {
  int format;               /* w4_format                                               */
  const uint8_t* packed;    /* [N][K/2]                                                 */
  const void* scales;       /* float absmax [N][K/bs] (NF4) or fp16 scale [N][K/gs] (INT4, FP4) */
  const float* codebook;    /* [16] for NF4, ignored otherwise                          */
  const uint16_t* x;        /* [M][K] fp16                                              */
  uint16_t* y;              /* [M][N] fp16                                              */
  int M, N, K, blocksize;
  int level;                /* dependency level, see above                              */
} w4_gemv_desc;

/* Validates every descriptor, then enqueues one GEMV launch per descriptor, in order, on `stream`
 * (each launch reads x after the previous one completed). */
int w4_gemv_sequence(const w4_gemv_desc* descs, int count, w4_stream_t stream);

/* Device workspace (bytes) that w4_step_create needs for `count` descriptors: one 32-bit counter
 * per level plus one, then (128-byte aligned) the persistent launch's tables: one TMA tensor map
 * per GEMV (128 bytes), the levels and the per-GEMV tiling (about 240 bytes per descriptor in
 * all). */
int64_t w4_step_workspace_bytes(int count);

/* A decode step captured once into a CUDA graph.  When every descriptor has the same format,
 * batch M <= 8 and (NF4) the same code book, the whole step is ONE persistent launch: every CTA
 * streams the weights of all levels ahead through its shared-memory ring and each level starts
 * reading x when the counters in `workspace` show the previous level complete.  Otherwise the
 * step is one launch per GEMV.  `workspace`: device memory of w4_step_workspace_bytes(count) bytes,
 * 16-byte aligned, owned by the caller, used only by this step; w4_step_create zeroes the
 * counters, writes the tables (and synchronises); every launch leaves the counters zero again and
 * only reads the tables.  Launches of one step must not overlap on
 * the GPU (stream order guarantees that).  The descriptors' pointers are baked into the graph:
 * the buffers must outlive the step.  No device memory is allocated. */
typedef struct w4_step w4_step;
int w4_step_create(const w4_gemv_desc* descs, int count, void* workspace, w4_step** out);
int w4_step_launch(w4_step* step, w4_stream_t stream);
int w4_step_destroy(w4_step* step);

/* w4_step_run_host -- one step with host buffers, all on `stream` and asynchronous: copies x_bytes
 * from x_host to the step's device input x_dev, launches the step, copies y_bytes from the step's
 * device output y_dev to y_host.  Host buffers should be pinned (page-locked) for the copies to
 * overlap; the caller synchronises `stream` before reading y_host.  x_bytes or y_bytes 0 skips that
 * copy.  Errors: W4_ERR_NULL (step, or a buffer of a non-empty copy), W4_ERR_SHAPE (negative
 * size), W4_ERR_CUDA. */
int w4_step_run_host(w4_step* step, const void* x_host, void* x_dev, int64_t x_bytes, void* y_host,
                     const void* y_dev, int64_t y_bytes, w4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * w4_gemv_levels_noalloc -- runs the descriptors as ONE persistent launch on `stream`, like
 * w4_step_create + w4_step_launch, without any device memory from the caller beyond its inputs
 * and outputs.  The pages have no counterpart of this entry point.  It is for callers that cannot
 * allocate device memory: code running inside a device-memory allocator or pool callback (a
 * cudaMalloc there re-enters the allocator), processes whose device memory a framework's caching
 * allocator has reserved up front (a cudaMalloc there fails or fragments the pool), serving loops
 * that forbid allocation after warm-up (cudaMalloc can synchronise the device and stall every
 * stream), and plugin interfaces that hand the callee only its input and output buffers.
 * The level counters and tables that w4_step_create keeps in a caller workspace live here in
 * fixed arrays inside libw4 (W4_NOALLOC_MAX_LEVELS + 1 32-bit words and about 61 KB of tables,
 * held on every GPU that loads the library until the process exits).  Limits: at most W4_NOALLOC_MAX_LEVELS levels and W4_NOALLOC_MAX_GEMVS
 * descriptors, else W4_ERR_LIMIT.  Same conditions as the single-launch step (one format,
 * M <= 8, one code book), else W4_ERR_UNSUPPORTED.  Each call first copies its tables in and
 * clears the counters it uses (an asynchronous copy from pageable host memory and a memset on
 * `stream`), then launches; it never calls cudaMalloc, cudaFree or any allocating routine.  The
 * first call on a device looks up the arrays' device addresses (cudaGetSymbolAddress) with that
 * device current and keeps them, with the id of the device's context; a later call in another
 * context (after cudaDeviceReset) looks them up again.  Make the first call in a context before
 * any stream capture.  Every call uses the same arrays,
 * so calls that overlap on the GPU (other streams, other host threads) race and give wrong
 * results: serialise them. */
#define W4_NOALLOC_MAX_LEVELS 256
#define W4_NOALLOC_MAX_GEMVS 256
int w4_gemv_levels_noalloc(const w4_gemv_desc* descs, int count, w4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Diagnostics. */
const char* w4_status_str(int status);
int w4_last_cuda_error(void);          /* cudaError_t of the last W4_ERR_CUDA in this thread */
/* Synchronises `stream`, reads and clears the device error word of the current device:
 * W4_OK, or W4_ERR_TIMEOUT if a bounded device-side wait ran out since the last check. */
int w4_device_check(w4_stream_t stream);
/* Kernel launches the library has issued in this process (for launch accounting). */
long long w4_launch_count(void);

/* Test hook for the timeout path.  The next GEMV launch in this process (small-batch or tcgen05
 * kernel, whichever the call dispatches to) has its weight producer issue no copies, so the bounded
 * waits (one second each) of the roles that depend on those copies run out; the kernel records the
 * failure, waits (bounded) for whatever copies and MMAs it did issue, frees its tensor memory and
 * returns without faulting.  Its output is garbage, and the next w4_device_check() returns
 * W4_ERR_TIMEOUT.  The context stays usable.  Returns W4_OK. */
int w4_inject_timeout_once(void);

#ifdef __cplusplus
}
#endif
#endif /* W4_H */
