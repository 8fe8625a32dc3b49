// w4_api.cu -- the C ABI of libw4 (include/w4.h): argument validation, dispatch, the decode-step
// sequence and its CUDA graph, diagnostics, and the NF4 code-book construction.
#include <atomic>
#include <cerrno>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/w4.h"
#include "w4_internal.h"

namespace w4 {

static std::atomic<long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<int> g_inject{0};
int take_fault_injection() { return g_inject.exchange(0); }

}  // namespace w4

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return W4_OK;
  t_last_cuda_error = static_cast<int>(e);
  return W4_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool pow2_in_range(int v) { return v >= 32 && v <= 256 && (v & (v - 1)) == 0; }

// Shape rules shared by every call on a packed matrix.
int check_shape(int N, int K, int bs) {
  if (!pow2_in_range(bs)) return W4_ERR_BLOCKSIZE;
  if (N < 1 || K < bs || K % bs != 0) return W4_ERR_SHAPE;
  if (K > W4_MAX_K) return W4_ERR_UNSUPPORTED;
  return W4_OK;
}

int check_gemv(int format, const uint8_t* packed, const void* scales, const float* codebook, const uint16_t* x,
               const uint16_t* y, int M, int N, int K, int bs) {
  if (format != W4_FMT_NF4 && format != W4_FMT_INT4 && format != W4_FMT_FP4) return W4_ERR_UNSUPPORTED;
  if (!packed || !scales || !x || !y || (format == W4_FMT_NF4 && !codebook)) return W4_ERR_NULL;
  int s = check_shape(N, K, bs);
  if (s != W4_OK) return s;
  if (M < 1) return W4_ERR_SHAPE;
  if (M > W4_MAX_BATCH) return W4_ERR_UNSUPPORTED;
  if (!aligned(packed, 16) || !aligned(scales, 16) || !aligned(x, 16) || !aligned(y, 2) ||
      (codebook && !aligned(codebook, 4)))
    return W4_ERR_ALIGN;
  return W4_OK;
}

// Batches above 8 go to the tcgen05 kernel (where it takes the shape); batches up to 8 stay on
// the small-batch kernel, the same kernel (and arithmetic, bit for bit) as the persistent step.
bool tc5_batch(int M) { return M > 8; }

// Largest batch one tensor-core launch takes with two accumulators; larger batches run as tiles of
// this many rows, or of twice as many (one 256-column accumulator) where the weight matrix alone
// has enough 128-row tiles to keep the SMs busy: each tile of weights is then decoded and read once
// per 256 batch rows instead of once per 128.
constexpr int kBatchTile = 128;

static bool wide_batch_tiles(int N) {
  const int nrb = (N + 127) / 128;
  return 2 * nrb > w4::device_sm_count();
}

int enqueue_gemv(int format, const uint8_t* packed, const void* scales, const float* codebook, const uint16_t* x,
                 uint16_t* y, int M, int N, int K, int bs, cudaStream_t stream);

// One batch tile of up to 256 rows on the tcgen05 kernel at 256 columns (above 128 rows), else as
// tiles of 128.
static int enqueue_wide_tile(int format, const uint8_t* packed, const void* scales, const float* codebook,
                             const uint16_t* x, uint16_t* y, int M, int N, int K, int bs, cudaStream_t stream) {
  if (M > kBatchTile) {
    cudaError_t e = w4::launch_gemv_tc5(format, packed, scales, codebook, reinterpret_cast<const __half*>(x),
                                        reinterpret_cast<__half*>(y), M, N, K, bs, true, stream);
    if (e != cudaErrorNotSupported) return cuda_status(e);
  }
  for (int m0 = 0; m0 < M; m0 += kBatchTile) {
    const int mm = (M - m0) < kBatchTile ? (M - m0) : kBatchTile;
    const int s = enqueue_gemv(format, packed, scales, codebook, x + (size_t)m0 * K, y + (size_t)m0 * N, mm, N, K,
                               bs, stream);
    if (s != W4_OK) return s;
  }
  return W4_OK;
}

// Enqueue one validated GEMV.  Batches above one launch's budget are split into launches over
// consecutive batch rows (each re-reads the weights): tiles of 128 or 256 rows, and within a tile
// the small-batch launches of at most 8 rows where the tensor cores do not serve.
int enqueue_gemv(int format, const uint8_t* packed, const void* scales, const float* codebook, const uint16_t* x,
                 uint16_t* y, int M, int N, int K, int bs, cudaStream_t stream) {
  if (M > kBatchTile) {
    const int tile = wide_batch_tiles(N) ? 2 * kBatchTile : kBatchTile;
    for (int m0 = 0; m0 < M; m0 += tile) {
      const int mm = (M - m0) < tile ? (M - m0) : tile;
      const int s = enqueue_wide_tile(format, packed, scales, codebook, x + (size_t)m0 * K, y + (size_t)m0 * N, mm,
                                      N, K, bs, stream);
      if (s != W4_OK) return s;
    }
    return W4_OK;
  }
  const __half* xh = reinterpret_cast<const __half*>(x);
  __half* yh = reinterpret_cast<__half*>(y);
  // batches above 8: the 5th-generation tensor cores (tcgen05; a batch below 16 is padded to 16
  // MMA columns at no extra MMA cost).  Batches up to 8 stay on the small-batch kernel, whose
  // arithmetic the persistent step kernel shares bit for bit.  Both batch >= 9 kernels need K to
  // be a multiple of 64; the mma.sync one (batch >= 32) also serves if the TMA descriptors cannot
  // be made.  Everything else runs as small-batch launches of at most 8 rows.
  if (tc5_batch(M)) {
    cudaError_t e = w4::launch_gemv_tc5(format, packed, scales, codebook, xh, yh, M, N, K, bs, true, stream);
    if (e != cudaErrorNotSupported) return cuda_status(e);
  }
  if (M >= 32) {
    cudaError_t e = w4::launch_gemv_tc(format, packed, scales, codebook, xh, yh, M, N, K, bs, true, stream);
    if (e != cudaErrorNotSupported) return cuda_status(e);
  }
  const int mb = w4::simt_max_batch(format, K, bs);
  if (mb < 1) return W4_ERR_UNSUPPORTED;
  for (int m0 = 0; m0 < M; m0 += mb) {
    const int mm = (M - m0) < mb ? (M - m0) : mb;
    cudaError_t e = w4::launch_gemv_simt(format, packed, scales, codebook, xh + (size_t)m0 * K,
                                         yh + (size_t)m0 * N, mm, N, K, bs, true, stream);
    if (e == cudaErrorNotSupported) return W4_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_status(e);
  }
  return W4_OK;
}

// Inverse of the standard normal CDF: Newton's method on Phi(x) - p with Phi(x) = erfc(-x/sqrt2)/2,
// started at 0.  For p in [1/2, 1) the iterates increase monotonically to the root (Phi is concave
// there), so the loop ends when a step no longer changes x.
double inv_norm_cdf_upper(double p) {
  const double kSqrt2 = 1.4142135623730951;
  const double kInvSqrt2Pi = 0.3989422804014327;
  double x = 0.0;
  for (int i = 0; i < 200; ++i) {
    const double f = 0.5 * std::erfc(-x / kSqrt2) - p;
    const double d = kInvSqrt2Pi * std::exp(-0.5 * x * x);
    const double nx = x - f / d;
    if (nx == x) break;
    x = nx;
  }
  return x;
}

}  // namespace

struct w4_step {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  long long kernels = 0;
};

extern "C" {

int w4_nf4_codebook(float out[16]) {
  if (!out) return W4_ERR_NULL;
  const double delta = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0));
  double v[16];
  int n = 0;
  for (int i = 0; i < 8; ++i) v[n++] = inv_norm_cdf_upper(delta + i * ((0.5 - delta) / 8.0));
  for (int i = 0; i < 7; ++i) v[n++] = -inv_norm_cdf_upper(delta + i * ((0.5 - delta) / 7.0));
  v[n++] = 0.0;
  // ascending order (insertion sort of 16 values)
  for (int i = 1; i < 16; ++i) {
    double t = v[i];
    int j = i - 1;
    while (j >= 0 && v[j] > t) { v[j + 1] = v[j]; --j; }
    v[j + 1] = t;
  }
  const double top = v[15];
  for (int i = 0; i < 16; ++i) out[i] = static_cast<float>(v[i] / top);
  return W4_OK;
}

int w4_quantize_nf4(const float* W, uint8_t* packed, float* absmax, const float* codebook, int N, int K,
                    int blocksize, w4_stream_t stream) {
  if (!W || !packed || !absmax || !codebook) return W4_ERR_NULL;
  int s = check_shape(N, K, blocksize);
  if (s != W4_OK) return s;
  if (!aligned(W, 16) || !aligned(packed, 16) || !aligned(absmax, 16) || !aligned(codebook, 4)) return W4_ERR_ALIGN;
  return cuda_status(w4::launch_quantize_nf4(W, packed, absmax, codebook, N, K, blocksize,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int w4_quantize_int4(const float* W, uint8_t* packed, uint16_t* scale, int N, int K, int group,
                     w4_stream_t stream) {
  if (!W || !packed || !scale) return W4_ERR_NULL;
  int s = check_shape(N, K, group);
  if (s != W4_OK) return s;
  if (!aligned(W, 16) || !aligned(packed, 16) || !aligned(scale, 16)) return W4_ERR_ALIGN;
  return cuda_status(w4::launch_quantize_int4(W, packed, reinterpret_cast<__half*>(scale), N, K, group,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int w4_quantize_fp4(const float* W, uint8_t* packed, uint16_t* scale, int N, int K, int group,
                    w4_stream_t stream) {
  if (!W || !packed || !scale) return W4_ERR_NULL;
  int s = check_shape(N, K, group);
  if (s != W4_OK) return s;
  if (!aligned(W, 16) || !aligned(packed, 16) || !aligned(scale, 16)) return W4_ERR_ALIGN;
  return cuda_status(w4::launch_quantize_fp4(W, packed, reinterpret_cast<__half*>(scale), N, K, group,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int w4_dequantize_nf4(const uint8_t* packed, const float* absmax, const float* codebook, float* W_out, int N,
                      int K, int blocksize, w4_stream_t stream) {
  if (!packed || !absmax || !codebook || !W_out) return W4_ERR_NULL;
  int s = check_shape(N, K, blocksize);
  if (s != W4_OK) return s;
  if (!aligned(W_out, 8) || !aligned(packed, 16) || !aligned(absmax, 16) || !aligned(codebook, 4)) return W4_ERR_ALIGN;
  return cuda_status(w4::launch_dequantize_nf4(packed, absmax, codebook, W_out, N, K, blocksize,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int w4_dequantize_int4(const uint8_t* packed, const uint16_t* scale, float* W_out, int N, int K, int group,
                       w4_stream_t stream) {
  if (!packed || !scale || !W_out) return W4_ERR_NULL;
  int s = check_shape(N, K, group);
  if (s != W4_OK) return s;
  if (!aligned(W_out, 8) || !aligned(packed, 16) || !aligned(scale, 16)) return W4_ERR_ALIGN;
  return cuda_status(w4::launch_dequantize_int4(packed, reinterpret_cast<const __half*>(scale), W_out, N, K, group,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

int w4_dequantize_fp4(const uint8_t* packed, const uint16_t* scale, float* W_out, int N, int K, int group,
                      w4_stream_t stream) {
  if (!packed || !scale || !W_out) return W4_ERR_NULL;
  int s = check_shape(N, K, group);
  if (s != W4_OK) return s;
  if (!aligned(W_out, 8) || !aligned(packed, 16) || !aligned(scale, 16)) return W4_ERR_ALIGN;
  return cuda_status(w4::launch_dequantize_fp4(packed, reinterpret_cast<const __half*>(scale), W_out, N, K, group,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int w4_gemv_nf4(const uint8_t* packed, const float* absmax, const float* codebook, const uint16_t* x, uint16_t* y,
                int M, int N, int K, int blocksize, w4_stream_t stream) {
  int s = check_gemv(W4_FMT_NF4, packed, absmax, codebook, x, y, M, N, K, blocksize);
  if (s != W4_OK) return s;
  return enqueue_gemv(W4_FMT_NF4, packed, absmax, codebook, x, y, M, N, K, blocksize,
                      reinterpret_cast<cudaStream_t>(stream));
}

int w4_gemv_int4(const uint8_t* packed, const uint16_t* scale, const uint16_t* x, uint16_t* y, int M, int N, int K,
                 int group, w4_stream_t stream) {
  int s = check_gemv(W4_FMT_INT4, packed, scale, nullptr, x, y, M, N, K, group);
  if (s != W4_OK) return s;
  return enqueue_gemv(W4_FMT_INT4, packed, scale, nullptr, x, y, M, N, K, group,
                      reinterpret_cast<cudaStream_t>(stream));
}

int w4_gemv_fp4(const uint8_t* packed, const uint16_t* scale, const uint16_t* x, uint16_t* y, int M, int N, int K,
                int group, w4_stream_t stream) {
  int s = check_gemv(W4_FMT_FP4, packed, scale, nullptr, x, y, M, N, K, group);
  if (s != W4_OK) return s;
  return enqueue_gemv(W4_FMT_FP4, packed, scale, nullptr, x, y, M, N, K, group,
                      reinterpret_cast<cudaStream_t>(stream));
}

static int check_descs(const w4_gemv_desc* descs, int count) {
  if (!descs) return W4_ERR_NULL;
  if (count < 1) return W4_ERR_SHAPE;
  int prev_level = 0;
  for (int i = 0; i < count; ++i) {
    const w4_gemv_desc& d = descs[i];
    int s = check_gemv(d.format, d.packed, d.scales, d.codebook, d.x, d.y, d.M, d.N, d.K, d.blocksize);
    if (s != W4_OK) return s;
    const int want_lo = (i == 0) ? 0 : prev_level;
    if (d.level < want_lo || d.level > (i == 0 ? 0 : prev_level + 1)) return W4_ERR_SHAPE;
    prev_level = d.level;
  }
  return W4_OK;
}

// The plan of one batch tile (M <= 256), validated arguments.
static int plan_tile(int format, int M, int N, int K, int blocksize, int sm_count, w4_gemv_plan_t* plan) {
  w4::Tc5Plan tp;
  if (tc5_batch(M) && w4::plan_tc5(M, N, K, blocksize, sm_count, &tp)) {
    *plan = w4_gemv_plan_t{W4_KERNEL_TCGEN05, 1, tp.nb, tp.threads, tp.smem, tp.ns, tp.grid, tp.ks};
    return W4_OK;
  }
  w4::SimtPlan sp;
  if (!w4::plan_simt(format, M, K, blocksize, &sp)) return W4_ERR_UNSUPPORTED;
  *plan = w4_gemv_plan_t{W4_KERNEL_SMALL_BATCH, sp.launches, sp.mb, sp.threads, sp.smem, sp.stages, 0, 1};
  return W4_OK;
}

int w4_gemv_plan(int format, int M, int N, int K, int blocksize, int sm_count, w4_gemv_plan_t* plan) {
  if (!plan) return W4_ERR_NULL;
  if (format != W4_FMT_NF4 && format != W4_FMT_INT4 && format != W4_FMT_FP4) return W4_ERR_UNSUPPORTED;
  int s = check_shape(N, K, blocksize);
  if (s != W4_OK) return s;
  if (M < 1 || sm_count < 1) return W4_ERR_SHAPE;
  if (M > W4_MAX_BATCH) return W4_ERR_UNSUPPORTED;
  if (M <= kBatchTile) return plan_tile(format, M, N, K, blocksize, sm_count, plan);
  // full tiles of 128 (or 256) rows, then the remainder tile; the figures are the full tile's
  w4::Tc5Plan wide;
  const int tile = 2 * ((N + 127) / 128) > sm_count && w4::plan_tc5(2 * kBatchTile, N, K, blocksize, sm_count, &wide)
                       ? 2 * kBatchTile
                       : kBatchTile;
  s = plan_tile(format, tile, N, K, blocksize, sm_count, plan);
  if (s != W4_OK) return s;
  plan->launches *= M / tile;
  if (M % tile) {
    w4_gemv_plan_t rest;
    s = plan_tile(format, M % tile, N, K, blocksize, sm_count, &rest);
    if (s != W4_OK) return s;
    plan->launches += rest.launches;
  }
  return W4_OK;
}

int w4_gemv_sequence(const w4_gemv_desc* descs, int count, w4_stream_t stream) {
  int s = check_descs(descs, count);
  if (s != W4_OK) return s;
  for (int i = 0; i < count; ++i) {
    const w4_gemv_desc& d = descs[i];
    s = enqueue_gemv(d.format, d.packed, d.scales, d.codebook, d.x, d.y, d.M, d.N, d.K, d.blocksize,
                     reinterpret_cast<cudaStream_t>(stream));
    if (s != W4_OK) return s;
  }
  return W4_OK;
}

// Step workspace: (count + 1) level counters, then, 128-byte aligned, the launch's device tables
// (a TMA tensor map, a level and a GEMV descriptor per descriptor; written once by w4_step_create,
// read by every launch).
static size_t ws_counter_bytes(int count) { return ((size_t)(count + 1) * 4 + 15) & ~(size_t)15; }

static void* ws_tables(void* workspace, int count) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(workspace) + ws_counter_bytes(count);
  return reinterpret_cast<void*>((a + 127) & ~(uintptr_t)127);
}

int64_t w4_step_workspace_bytes(int count) {
  if (count < 1 || count > w4::kStepMaxGemvs) return count < 1 ? 0 : ((int64_t)(count + 1) * 4 + 255) / 256 * 256;
  return ((int64_t)ws_counter_bytes(count) + 128 + (int64_t)w4::step_tables_bytes(count) + 255) / 256 * 256;
}

// True when the step can run as one persistent launch of the small-batch kernel.
static bool step_is_persistent(const w4_gemv_desc* descs, int count) {
  if (count > w4::kStepMaxGemvs) return false;
  for (int i = 0; i < count; ++i) {
    const w4_gemv_desc& d = descs[i];
    if (d.format != descs[0].format || d.M != descs[0].M || d.M > 8) return false;
    if (d.format == W4_FMT_NF4 && d.codebook != descs[0].codebook) return false;
    if (w4::simt_max_batch(d.format, d.K, d.blocksize) < d.M) return false;
  }
  return true;
}

int w4_step_create(const w4_gemv_desc* descs, int count, void* workspace, w4_step** out) {
  if (!out) return W4_ERR_NULL;
  *out = nullptr;
  int s = check_descs(descs, count);
  if (s != W4_OK) return s;
  const bool persistent = step_is_persistent(descs, count);
  if (persistent && !workspace) return W4_ERR_NULL;
  if (workspace && !aligned(workspace, 16)) return W4_ERR_ALIGN;
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_status(e);
  std::vector<w4::StepJob> jobs;
  if (persistent) {
    jobs.resize((size_t)count);
    for (int i = 0; i < count; ++i) {
      const w4_gemv_desc& d = descs[i];
      jobs[i] = w4::StepJob{d.packed, d.scales, reinterpret_cast<const __half*>(d.x), reinterpret_cast<__half*>(d.y),
                            d.N, d.K, d.blocksize, d.level};
    }
    // counters zeroed, tables written once, before the capture
    std::vector<uint8_t> blob(w4::step_tables_bytes(count));
    e = w4::step_simt_tables(descs[0].format, jobs.data(), count, descs[0].M, ws_tables(workspace, count),
                             blob.data());
    if (e == cudaErrorNotSupported) {
      cudaStreamDestroy(cs);
      return W4_ERR_UNSUPPORTED;
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, (size_t)w4_step_workspace_bytes(count), cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws_tables(workspace, count), blob.data(), blob.size(), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) {
      cudaStreamDestroy(cs);
      return cuda_status(e);
    }
  }
  w4_step* st = new w4_step();
  const long long before = w4::g_launches.load();
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    if (persistent) {
      cudaError_t e3 = w4::launch_step_simt(descs[0].format, jobs.data(), count, descs[0].M, descs[0].codebook,
                                            reinterpret_cast<unsigned*>(workspace), ws_tables(workspace, count), true, cs);
      if (e3 != cudaSuccess) s = (e3 == cudaErrorNotSupported) ? W4_ERR_UNSUPPORTED : cuda_status(e3);
    } else {
      for (int i = 0; i < count && s == W4_OK; ++i) {
        const w4_gemv_desc& d = descs[i];
        s = enqueue_gemv(d.format, d.packed, d.scales, d.codebook, d.x, d.y, d.M, d.N, d.K, d.blocksize, cs);
      }
    }
    cudaError_t e2 = cudaStreamEndCapture(cs, &st->graph);
    if (e == cudaSuccess) e = e2;
  }
  // launches recorded during capture are not executions; count them per replay instead
  st->kernels = w4::g_launches.load() - before;
  w4::g_launches.fetch_sub(st->kernels);
  if (e == cudaSuccess && s == W4_OK) e = cudaGraphInstantiate(&st->exec, st->graph, 0);
  cudaStreamDestroy(cs);
  if (s != W4_OK || e != cudaSuccess) {
    if (st->exec) cudaGraphExecDestroy(st->exec);
    if (st->graph) cudaGraphDestroy(st->graph);
    delete st;
    return s != W4_OK ? s : cuda_status(e);
  }
  *out = st;
  return W4_OK;
}

int w4_gemv_levels_noalloc(const w4_gemv_desc* descs, int count, w4_stream_t stream) {
  int s = check_descs(descs, count);
  if (s != W4_OK) return s;
  const int nlevels = descs[count - 1].level + 1;
  if (count > W4_NOALLOC_MAX_GEMVS || nlevels > W4_NOALLOC_MAX_LEVELS || nlevels > w4::noalloc_max_levels())
    return W4_ERR_LIMIT;
  if (!step_is_persistent(descs, count)) return W4_ERR_UNSUPPORTED;
  w4::StepJob jobs[W4_NOALLOC_MAX_GEMVS];
  for (int i = 0; i < count; ++i) {
    const w4_gemv_desc& d = descs[i];
    jobs[i] = w4::StepJob{d.packed, d.scales, reinterpret_cast<const __half*>(d.x), reinterpret_cast<__half*>(d.y),
                          d.N, d.K, d.blocksize, d.level};
  }
  cudaError_t e = w4::launch_step_simt_noalloc(descs[0].format, jobs, count, descs[0].M, descs[0].codebook, nlevels,
                                               reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return W4_ERR_UNSUPPORTED;
  return cuda_status(e);
}

int w4_step_launch(w4_step* step, w4_stream_t stream) {
  if (!step || !step->exec) return W4_ERR_NULL;
  cudaError_t e = cudaGraphLaunch(step->exec, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) w4::g_launches.fetch_add(step->kernels);
  return cuda_status(e);
}

int w4_step_run_host(w4_step* step, const void* x_host, void* x_dev, int64_t x_bytes, void* y_host,
                     const void* y_dev, int64_t y_bytes, w4_stream_t stream) {
  if (!step || !step->exec) return W4_ERR_NULL;
  if (x_bytes < 0 || y_bytes < 0) return W4_ERR_SHAPE;
  if ((x_bytes > 0 && (!x_host || !x_dev)) || (y_bytes > 0 && (!y_host || !y_dev))) return W4_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (x_bytes > 0) e = cudaMemcpyAsync(x_dev, x_host, (size_t)x_bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaGraphLaunch(step->exec, s);
  if (e != cudaSuccess) return cuda_status(e);
  w4::g_launches.fetch_add(step->kernels);
  if (y_bytes > 0) e = cudaMemcpyAsync(y_host, y_dev, (size_t)y_bytes, cudaMemcpyDeviceToHost, s);
  return cuda_status(e);
}

int w4_step_destroy(w4_step* step) {
  if (!step) return W4_ERR_NULL;
  if (step->exec) cudaGraphExecDestroy(step->exec);
  if (step->graph) cudaGraphDestroy(step->graph);
  delete step;
  return W4_OK;
}

const char* w4_status_str(int status) {
  switch (status) {
    case W4_OK: return "ok";
    case W4_ERR_NULL: return "null pointer";
    case W4_ERR_SHAPE: return "bad shape";
    case W4_ERR_ALIGN: return "misaligned pointer";
    case W4_ERR_BLOCKSIZE: return "block size must be a power of two in [32, 256]";
    case W4_ERR_CUDA: return "CUDA runtime error";
    case W4_ERR_TIMEOUT: return "device-side wait timed out";
    case W4_ERR_UNSUPPORTED: return "unsupported by this build";
    case W4_ERR_LIMIT: return "beyond the fixed counter array of w4_gemv_levels_noalloc (256 levels, 256 GEMVs)";
    default: return "unknown status";
  }
}

int w4_last_cuda_error(void) { return t_last_cuda_error; }

int w4_device_check(w4_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  // every translation unit's copy of the error word: the small-batch and the tensor-core kernels
  const unsigned int v = w4::read_clear_error_persist() | w4::read_clear_error_tc5();
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  return v ? W4_ERR_TIMEOUT : W4_OK;
}

long long w4_launch_count(void) { return w4::g_launches.load(); }

int w4_inject_timeout_once(void) {
  w4::g_inject.store(1);
  return W4_OK;
}

}  // extern "C"
