// w4_gemv.cu -- fused 4-bit dequant-GEMV on CUDA cores for batches 1 ... 31 (sm_103a).
//
// What it computes ("LLM Quantization on RTX 4060: Where 4-bit Decode Falls Behind FP16",
// sections "Fused Kernel: Moving Dequantization On-Chip" and "Kernel Implementation"):
//   y[m][n] = sum_k w_hat[n][k] * x[m][k], w_hat decoded on chip from the packed nibbles and the
//   block scale, FP32 accumulation, FP16 result; no dequantised matrix ever reaches DRAM.
//
// How it maps to GB300:
//   * A persistent grid (two CTAs per SM) walks tiles of whole rows.  One producer warp streams
//     each tile's packed bytes and scales into a 4-stage shared-memory ring with 1-D bulk async
//     copies (the TMA unit), completion tracked by mbarriers; consumers release a stage with an
//     mbarrier arrive.  Rows are contiguous, so one tile is one copy.
//   * Each consumer thread owns one 32-weight column chunk (16 packed bytes) of every row it
//     touches, so its slice of x lives in registers for the whole kernel; a tile's rows are swept
//     by all consumer threads, and the per-row partial sums are reduced through shared memory in a
//     fixed order (the warp-shuffle-then-shared-memory idiom of "Do Quantization and Sparsity make
//     LLM Inference Faster ?", section "Optional: what does the custom kernel actually do?").
//   * NF4 decode: a 256-entry table indexed by a whole packed byte returns both code values as one
//     half2 (the code book rounded to FP16); it is replicated once per lane with lane-private banks,
//     so lookups never conflict.  Products are formed with mixed-precision FMAs (FP16 x FP16 -> FP32,
//     exact) and summed in FP32; the FP32 absmax multiplies each 32-weight partial.
//   * INT4 decode: x is converted once per thread to 16-bit fixed point with one exponent per
//     32-weight chunk (X = x * 2^(15-E), exact for the chunk's large entries), split into a signed
//     high byte and an unsigned low byte; the nibbles are isolated as bytes and multiplied with
//     dp4a (4 MACs per instruction).  sum (q-8) x = 2^(E-15) (sum q X - 8 sum X), scaled by s.
//   * Programmatic dependent launch: the producer prefetches weights and scales and the consumers
//     build the lookup table before griddepcontrol.wait; x is read and y written after it.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4_common.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr int kStages = 4;
constexpr int kMaxConsumers = 320;      // consumer threads: one per chunk of a row, times rows per sweep
constexpr int kLutBytes = 256 * 32 * 4; // NF4 byte-pair table, one copy per lane

struct GemvParams {
  const uint8_t* packed;
  const void* scales;
  const float* codebook;
  const __half* x;
  __half* y;
  int M, N, K, bs;
  int cpr;              // chunks (16 packed bytes) per row = K / 32
  int rps;              // rows per sweep = consumer threads / cpr
  int n_consumer_warps;
  int rpt;              // rows per tile
  int n_tiles;
  int srb;              // scale bytes per row
  int stage_w;          // bytes of one packed stage (rpt * K / 2)
  int stage_s;          // bytes of one scale stage (rpt * srb rounded up to 16)
  int red_floats;       // floats of one partial-sum buffer
  int inject_timeout;   // test hook: the producer issues nothing, so the consumers' waits run out
};

// Shared-memory layout offsets (bytes), identical on host and device.
struct SmemLayout {
  int lut, w, s, red, bar, total;
};

__host__ __device__ inline SmemLayout smem_layout(int format, int MB, const GemvParams& p) {
  SmemLayout L;
  int off = 0;
  L.lut = off;
  if (format == 0) off += kLutBytes;
  L.w = off;
  off += kStages * p.stage_w;
  L.s = off;
  off += kStages * p.stage_s;
  L.red = off;
  off += 2 * p.red_floats * 4;
  off = (off + 15) & ~15;
  L.bar = off;
  off += 2 * kStages * 8;
  L.total = off;
  (void)MB;
  return L;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// acc += lo(c) * lo(x) + hi(c) * hi(x), products exact (FP16 x FP16 fits FP32), FP32 sums.
__device__ __forceinline__ void mixed_dot2(float& acc, uint32_t c2, uint32_t x2) {
  asm("{\n .reg .f16 c0, c1, x0, x1;\n"
      " mov.b32 {c0, c1}, %1;\n mov.b32 {x0, x1}, %2;\n"
      " fma.rn.f32.f16 %0, c0, x0, %0;\n fma.rn.f32.f16 %0, c1, x1, %0;\n}"
      : "+f"(acc) : "r"(c2), "r"(x2));
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Per-thread view of x for its chunk: NF4 keeps 16 half2 pairs per batch row; INT4 keeps 16
// digit words per batch row (hi/lo bytes of X for odd and even elements of each packed word),
// the chunk exponent factor 2^(E-15) and 8 * sum(X).
template <int FMT, int MB>
struct XSlice {
  uint32_t v[MB][16];
  float f[MB];
  int s8[MB];
};

template <int FMT, int MB>
__device__ __forceinline__ void load_x_slice(XSlice<FMT, MB>& xs, const __half* __restrict__ x, int M, int K,
                                             int chunk) {
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    uint32_t h[16];
    if (m < M) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)m * K + (size_t)chunk * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 q = src[i];
        h[4 * i + 0] = q.x; h[4 * i + 1] = q.y; h[4 * i + 2] = q.z; h[4 * i + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = 0u;
    }
    if (FMT == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) xs.v[m][i] = h[i];
      xs.f[m] = 1.0f;
      xs.s8[m] = 0;
    } else {
      // element e of the chunk: half number e of the 16 registers
      float xf[32];
      float mx = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __half2 hh = *reinterpret_cast<__half2*>(&h[i]);
        float2 f2 = __half22float2(hh);
        xf[2 * i] = f2.x;
        xf[2 * i + 1] = f2.y;
        mx = fmaxf(mx, fmaxf(fabsf(f2.x), fabsf(f2.y)));
      }
      int E = 0;
      (void)frexpf(mx, &E);                 // mx < 2^E (mx == 0 gives E = 0)
      const float up = ldexpf(1.0f, 15 - E);
      int X[32];
      int sx = 0;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        X[e] = __float2int_rn(xf[e] * up);  // exact for |x| >= 2^(E-5); |X| <= 32752
        sx += X[e];
      }
      // packed word i holds elements 8i..8i+7; lo nibbles -> elements 8i+1,3,5,7; hi -> 8i+0,2,4,6
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ho = 0, lo = 0, he = 0, le = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int eo = 8 * i + 2 * b + 1, ee = 8 * i + 2 * b;
          ho |= (uint32_t)((X[eo] >> 8) & 0xff) << (8 * b);
          lo |= (uint32_t)(X[eo] & 0xff) << (8 * b);
          he |= (uint32_t)((X[ee] >> 8) & 0xff) << (8 * b);
          le |= (uint32_t)(X[ee] & 0xff) << (8 * b);
        }
        xs.v[m][4 * i + 0] = ho;
        xs.v[m][4 * i + 1] = lo;
        xs.v[m][4 * i + 2] = he;
        xs.v[m][4 * i + 3] = le;
      }
      xs.f[m] = ldexpf(1.0f, E - 15);
      xs.s8[m] = 8 * sx;
    }
  }
}

template <int FMT, int MB>
__global__ void __launch_bounds__(kMaxConsumers + 32, 1) gemv_simt_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout L = smem_layout(FMT, MB, p);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* empty = full + kStages;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_cons = p.n_consumer_warps * 32;
  const bool producer = (warp == p.n_consumer_warps);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], p.n_consumer_warps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (producer) {
    // ------------------------------------------------------------------ producer warp
    if (p.inject_timeout) return;   // nothing issued, nothing in flight
    const uint64_t pol = policy_evict_first();
    int j = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++j) {
      const int st = j % kStages;
      const int round = j / kStages;
      // The first kStages tiles are prefetched while the previous kernel in the stream may still be
      // running.  Before waiting on the consumers, wait for that kernel: the consumers cannot start
      // before it completes, so only from here on is a long wait a lost wait.
      if (round == 1 && st == 0) pdl_wait();
      if (round > 0 && ok) ok = mbar_wait(&empty[st], (round - 1) & 1, 0x101);
      const int r0 = tile * p.rpt;
      const int nrows = min(p.rpt, p.N - r0);
      const uint32_t wbytes = (uint32_t)nrows * (uint32_t)(p.K / 2);
      const uint32_t sbytes = (uint32_t)nrows * (uint32_t)p.srb;
      const uint32_t sbulk = sbytes & ~15u;
      uint8_t* dst_w = smem + L.w + st * p.stage_w;
      uint8_t* dst_s = smem + L.s + st * p.stage_s;
      const uint8_t* src_s = reinterpret_cast<const uint8_t*>(p.scales) + (size_t)r0 * p.srb;
      if (lane == 0) {
        if (ok) {
          // scale bytes that do not fill a 16-byte unit at the end of the matrix: plain copies
          for (uint32_t b = sbulk; b < sbytes; ++b) dst_s[b] = src_s[b];
          mbar_arrive_expect_tx(&full[st], wbytes + sbulk);
          bulk_g2s(dst_w, p.packed + (size_t)r0 * (p.K / 2), wbytes, &full[st], pol);
          if (sbulk) bulk_g2s(dst_s, src_s, sbulk, &full[st], pol);
        } else {
          mbar_arrive(&full[st]);   // keep the consumers' phase count moving after a timeout
        }
      }
      __syncwarp();
    }
    // Do not leave while bulk copies into this CTA's shared memory may still be in flight.
    if (lane == 0) {
      const int issued = j;
      for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k) {
        mbar_wait(&full[k % kStages], (k / kStages) & 1, 0x102);
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumer threads
  const int t = threadIdx.x;
  const int rho = t / p.cpr;
  const int chunk = t - rho * p.cpr;
  const bool active = rho < p.rps;
  const uint32_t lut_lane = smem_u32(smem + L.lut) + (uint32_t)lane * 4u;

  if (FMT == 0) {
    // byte-pair table: entry b = half2(fp16(code[b >> 4]), fp16(code[b & 15])), one copy per lane
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + L.lut);
    for (int i = t; i < 256 * 32; i += n_cons) {
      const int b = i >> 5;
      const __half lo = __float2half_rn(__ldg(p.codebook + (b >> 4)));
      const __half hi = __float2half_rn(__ldg(p.codebook + (b & 15)));
      lut[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(n_cons) : "memory");

  pdl_wait();   // x may be produced by the previous kernel in the stream

  XSlice<FMT, MB> xs;
  if (active) load_x_slice<FMT, MB>(xs, p.x, p.M, p.K, chunk);

  float* red_base = reinterpret_cast<float*>(smem + L.red);
  const int K2 = p.K / 2;
  int j = 0;
  bool ok = true;
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x, ++j) {
    const int st = j % kStages;
    if (ok) ok = mbar_wait(&full[st], (j / kStages) & 1, 0x103);
    const int r0 = tile * p.rpt;
    const int nrows = min(p.rpt, p.N - r0);
    const uint32_t sw = smem_u32(smem + L.w + st * p.stage_w);
    const uint32_t ss = smem_u32(smem + L.s + st * p.stage_s);
    float* red = red_base + (j & 1) * p.red_floats;
    if (active && ok) {
      for (int lr = rho; lr < nrows; lr += p.rps) {
        const uint4 wv = lds128(sw + (uint32_t)(lr * K2 + chunk * 16));
        float part[MB];
        if (FMT == 0) {
          const float a = __uint_as_float(lds32(ss + (uint32_t)(lr * p.srb + ((chunk * 32) / p.bs) * 4)));
          float acc[MB];
#pragma unroll
          for (int m = 0; m < MB; ++m) acc[m] = 0.0f;
          const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              uint32_t byte;
              asm("prmt.b32 %0, %1, 0, %2;" : "=r"(byte) : "r"(w4[i]), "r"(0x4440 + b));
              const uint32_t c2 = lds32(lut_lane + byte * 128u);
#pragma unroll
              for (int m = 0; m < MB; ++m) mixed_dot2(acc[m], c2, xs.v[m][4 * i + b]);
            }
          }
#pragma unroll
          for (int m = 0; m < MB; ++m) part[m] = acc[m] * a;
        } else {
          const uint32_t sh = lds_u16(ss + (uint32_t)(lr * p.srb + ((chunk * 32) / p.bs) * 2));
          const float s = __half2float(__ushort_as_half((unsigned short)sh));
          int ah[MB], al[MB];
#pragma unroll
          for (int m = 0; m < MB; ++m) { ah[m] = 0; al[m] = 0; }
          const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t lo = w4[i] & 0x0f0f0f0fu;
            const uint32_t hi = (w4[i] >> 4) & 0x0f0f0f0fu;
#pragma unroll
            for (int m = 0; m < MB; ++m) {
              ah[m] = dp4a_us(lo, xs.v[m][4 * i + 0], ah[m]);
              al[m] = dp4a_uu(lo, xs.v[m][4 * i + 1], al[m]);
              ah[m] = dp4a_us(hi, xs.v[m][4 * i + 2], ah[m]);
              al[m] = dp4a_uu(hi, xs.v[m][4 * i + 3], al[m]);
            }
          }
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            const int tot = ah[m] * 256 + al[m] - xs.s8[m];
            part[m] = (float)tot * (s * xs.f[m]);
          }
        }
#pragma unroll
        for (int m = 0; m < MB; ++m) red[(m * p.rpt + lr) * p.cpr + chunk] = part[m];
      }
    }
    // stage fully read by this warp -> release it to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons) : "memory");
    // reduce: one warp per output, lanes over the row's chunks, fixed order
    const int outs = nrows * MB;
    for (int o = warp; o < outs; o += p.n_consumer_warps) {
      const int m = o / nrows;
      const int lr = o - m * nrows;
      const float* rr = red + (m * p.rpt + lr) * p.cpr;
      float v = 0.0f;
      for (int c = lane; c < p.cpr; c += 32) v += rr[c];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0 && m < p.M) p.y[(size_t)m * p.N + r0 + lr] = __float2half_rn(v);
    }
  }
}

static int g_sm_count = 0;

int device_sm_count() {
  if (g_sm_count == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (g_sm_count <= 0) g_sm_count = 1;
  }
  return g_sm_count;
}

static int gcd_int(int a, int b) {
  while (b) { int t = a % b; a = b; b = t; }
  return a;
}

template <int FMT, int MB>
static cudaError_t launch_mb(GemvParams p, int smem, int align_rows, bool pdl, cudaStream_t stream) {
  auto kern = gemv_simt_kernel<FMT, MB>;
  static bool attr_done = false;   // one flag per template instance
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int threads = p.n_consumer_warps * 32 + 32;
  // resident CTAs per SM for this block size and shared-memory footprint (cached per instance)
  static int occ_threads = -1, occ_smem = -1, occ_val = 1;
  if (occ_threads != threads || occ_smem != smem) {
    int v = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, (size_t)smem);
    if (e != cudaSuccess) return e;
    occ_threads = threads; occ_smem = smem; occ_val = v < 1 ? 1 : (v > 2 ? 2 : v);
  }
  const int gmax = device_sm_count() * occ_val;
  // balanced tiling: every CTA gets the same number of tiles (the last few may get one less)
  const int tiles_per_cta = (p.N + gmax * p.rpt - 1) / (gmax * p.rpt);
  int rpt = (p.N + gmax * tiles_per_cta - 1) / (gmax * tiles_per_cta);
  rpt = ((rpt + align_rows - 1) / align_rows) * align_rows;
  if (rpt > p.rpt) rpt = p.rpt;
  p.rpt = rpt;
  p.n_tiles = (p.N + rpt - 1) / rpt;
  const int grid = (p.n_tiles + tiles_per_cta - 1) / tiles_per_cta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  return e;
}

// Host-side plan of one launch: everything but the balanced tiling, which depends on occupancy.
static bool plan_simt(int format, int M, int N, int K, int bs, GemvParams& p, int& align_rows, int& MB,
                      SmemLayout& L) {
  p.M = M; p.N = N; p.K = K; p.bs = bs;
  p.cpr = K / 32;
  if (p.cpr > kMaxConsumers || M < 1 || M > 8) return false;
  const int target_threads = 288;
  p.rps = p.cpr >= target_threads ? 1 : target_threads / p.cpr;
  p.n_consumer_warps = (p.rps * p.cpr + 31) / 32;
  const int es = (format == 0) ? 4 : 2;
  p.srb = (K / bs) * es;
  // rows per tile: at most about 14 KB of packed bytes per stage, and a multiple of the row count
  // that keeps every tile's scale copy 16-byte aligned
  align_rows = 16 / gcd_int(p.srb, 16);
  int rpt_max = 14336 / (K / 2);
  if (rpt_max < 1) rpt_max = 1;
  rpt_max = ((rpt_max + align_rows - 1) / align_rows) * align_rows;
  p.rpt = rpt_max;
  p.n_tiles = 0;                    // set by launch_mb from the balanced tiling
  p.stage_w = rpt_max * (K / 2);
  p.stage_s = ((rpt_max * p.srb) + 15) & ~15;
  MB = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
  p.red_floats = MB * rpt_max * p.cpr;
  L = smem_layout(format, MB, p);
  return L.total <= 227 * 1024;
}

int simt_max_batch(int format, int K, int bs) {
  GemvParams p{};
  SmemLayout L;
  int align_rows, MB;
  for (int m : {8, 4, 2, 1}) {
    if (plan_simt(format, m, 1, K, bs, p, align_rows, MB, L)) return m;
  }
  return 0;
}

cudaError_t launch_gemv_simt(int format, const uint8_t* packed, const void* scales, const float* codebook,
                             const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                             cudaStream_t stream) {
  GemvParams p{};
  p.inject_timeout = 0;
  int align_rows = 1, MB = 1;
  SmemLayout L;
  if (!plan_simt(format, M, N, K, bs, p, align_rows, MB, L)) return cudaErrorNotSupported;
  p.packed = packed; p.scales = scales; p.codebook = codebook; p.x = x; p.y = y;
  p.inject_timeout = take_fault_injection();
  if (format == 0) {
    switch (MB) {
      case 1: return launch_mb<0, 1>(p, L.total, align_rows, pdl, stream);
      case 2: return launch_mb<0, 2>(p, L.total, align_rows, pdl, stream);
      case 4: return launch_mb<0, 4>(p, L.total, align_rows, pdl, stream);
      default: return launch_mb<0, 8>(p, L.total, align_rows, pdl, stream);
    }
  } else {
    switch (MB) {
      case 1: return launch_mb<1, 1>(p, L.total, align_rows, pdl, stream);
      case 2: return launch_mb<1, 2>(p, L.total, align_rows, pdl, stream);
      case 4: return launch_mb<1, 4>(p, L.total, align_rows, pdl, stream);
      default: return launch_mb<1, 8>(p, L.total, align_rows, pdl, stream);
    }
  }
}

unsigned int read_clear_error_gemv() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v));
  cudaMemcpyToSymbol(g_error_word, &z, sizeof(z));
  return v;
}

}  // namespace w4
