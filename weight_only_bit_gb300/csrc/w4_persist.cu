// w4_persist.cu -- fused 4-bit dequant-GEMV on CUDA cores (batches 1 ... 31), one persistent,
// warp-specialised kernel for a single GEMV or for every GEMV of a decode step (sm_103a).
//
// Computes y[m][n] = sum_k w_hat[n][k] * x[m][k] with w_hat decoded on chip, FP32 accumulation and
// an FP16 result; no dequantised matrix ever reaches DRAM ("LLM Quantization on RTX 4060: Where
// 4-bit Decode Falls Behind FP16", sections "Fused Kernel: Moving Dequantization On-Chip" and
// "Kernel Implementation").
//
// Work: each GEMV is cut into tiles of whole rows (rows are contiguous in memory, so a tile is one
// span).  GEMVs are grouped into levels; a level's GEMVs are independent of each other (the
// projections of one decode layer that read the same activation: q, k, v / o / gate, up / down).
// A level's x is read only after every tile of the previous level is complete, which models the
// decode step's data dependencies ("Do Quantization and Sparsity make LLM Inference Faster ?",
// section "What we did": the 197 GEMVs of one step).  Level 0 waits for the previous kernel in the
// stream (programmatic dependent launch); later levels wait on tile counters in global memory.
// Tile t of a level goes to CTA t mod gridDim.x; the grid is one CTA per SM, all co-resident.
//
// Roles in a CTA:
//   * producer warp: streams each tile's packed bytes and scales into a shared-memory ring of up to
//     eight stages with 1-D bulk async copies (TMA unit), mbarrier completion and an L2 evict-first
//     hint.  Weights never depend on other GEMVs, so it runs ahead across level boundaries and
//     prefetches later levels.  It issues copies only while its consumers compute (a stream gate
//     opened once a level's x is loaded and closed when the CTA's last tile of the level is
//     reduced): DRAM traffic during the grid-wide wait between levels multiplies that wait.  At
//     most three copies are in flight, which already saturates DRAM;
//   * consumer warps: thread (rho, chunk) owns one 32-weight column chunk, loads that slice of x
//     (through L1, which merges the requests of the threads sharing it) into registers for the
//     whole level, and produces one partial sum per (row, chunk), two rows at a time, into one of
//     two partial-sum buffers;
//   * reducer warp: sums each row's partials in a fixed order (eight interleaved sequences, then a
//     fixed tree, over 1, 2, 4 or 8 lanes per row with warp shuffles: the reduction idiom of "Do
//     Quantization and Sparsity make LLM Inference Faster ?", "Optional: what does the custom
//     kernel actually do?"), writes y, and after the CTA's last tile of a level publishes
//     completion with one release.  The order depends only on K, so a row gets the same bits
//     whatever the tiling.  Each lane issues a whole batch of loads before its first add: the
//     shared-memory queue is long while consumers decode, so one round trip per tile, not one per
//     partial, keeps the reducer ahead of the consumers.
// Every wait is bounded in wall-clock time; a lost wait is recorded in the device error word and
// the kernel runs to its end without further waiting.
#include <cstdint>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4_common.cuh"
#include "w4_decode.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr int kMaxStages = 8;
constexpr int kMaxInFlight = 3;         // copies outstanding per CTA: enough for full DRAM bandwidth
constexpr int kMaxConsumers = 320;      // longest row served: 320 chunks (K = 10240)
constexpr int kStageTarget = 65536;     // packed bytes per stage (about): large tiles amortise each
                                        // tile's barrier round trips; smaller when the ring won't fit
constexpr int kRedBufs = 2;             // partial-sum buffers: the reducer may lag one tile
constexpr int kRedCapFloats = 8192;     // largest partial-sum buffer (floats)
constexpr int kXDigitCap = 40960;       // largest INT4 x digit table shared in shared memory (bytes)
constexpr int kSmemCap = 227 * 1024;

// Consumer warps per CTA by batch block: as many as the registers of one SM allow.
__host__ __device__ constexpr int cons_warps(int MB) { return MB <= 1 ? 18 : MB == 2 ? 16 : 10; }

// Lanes of the reducer warp per output row: all of a tile's outputs in one pass when possible.
__host__ __device__ inline int red_lanes(int outs) {
  int q = 8;
  while (q > 1 && outs * q > 32) q >>= 1;
  return q;
}

// Row stride (floats) of a partial-sum buffer: at least cpr and an odd multiple of Q, so the
// (row, lane) reads of one reducer pass fall in 32 distinct banks.
__host__ __device__ inline int red_stride(int cpr, int Q) { return cpr + ((Q - cpr) & (2 * Q - 1)); }

struct PGemv {
  const uint8_t* packed;
  const void* scales;
  const __half* x;
  __half* y;
  int N, K, bs, rpt;       // rpt: rows per tile
  int tile0, ntiles, srb;  // global tile range; scale bytes per row
  int cpr;                 // chunks per row (K / 32)
};

struct PLevel {
  int gemv0, ngemv, tile0, ntiles;
};

template <int MAXL, int MAXG>
struct PParams {
  const float* codebook;
  unsigned int* counters;  // [nlevels + 1] when nlevels > 1, else null
  int nlevels, ngemvs, M, inject_timeout;
  int stages, stage_w, stage_s, red_floats, n_consumer_warps;
  int xd_bytes;            // INT4: shared x digit table (0: every thread converts its slice)
  PLevel lv[MAXL];
  PGemv gm[MAXG];
};

struct PLayout {
  int lut, xd, w, s, red, bar, total;
};

__host__ __device__ inline PLayout playout(int fmt, int stages, int stage_w, int stage_s, int red_floats,
                                           int xd_bytes) {
  PLayout L;
  int off = 0;
  L.lut = 0;
  if (fmt == 0) off += kLutBytes;
  L.xd = off;
  off += (xd_bytes + 15) & ~15;   // bulk copies into the ring need 16-byte alignment
  L.w = off;
  off += stages * stage_w;
  L.s = off;
  off += stages * stage_s;
  L.red = off;
  off += kRedBufs * red_floats * 4;
  off = (off + 15) & ~15;
  L.bar = off;
  off += (2 * kMaxStages + 2 * kRedBufs) * 8 + 16;   // ring and buffer barriers, then the gate
  L.total = off;
  return L;
}

__device__ __forceinline__ int first_owned(int tile0) {
  const int G = (int)gridDim.x;
  const int b = (int)blockIdx.x;
  return tile0 + (((b - tile0) % G) + G) % G;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Adds v with release semantics at GPU scope: every write ordered before it (this thread's, and
// its warp's through a preceding __syncwarp) is visible to a thread that acquires the new value.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *p >= target (other CTAs' releases).  Polls back to back for the first
// 20 microseconds, then backs off.  Records `site` on timeout.
__device__ __forceinline__ bool wait_counter(const unsigned* p, unsigned target, uint32_t site) {
  if (ld_acquire_u32(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (ld_acquire_u32(p) >= target) return true;
    const uint64_t dt = globaltimer_ns() - t0;
    if (dt > kWaitLimitNs) break;
    if (dt > 20000) __nanosleep(256);
  }
  atomicCAS(&g_error_word, 0u, site);
  return false;
}

// Bounded wait until the stream gate is open.
__device__ __forceinline__ bool wait_gate(volatile int* gate, uint32_t site) {
  if (*gate) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(64);
    if (*gate) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  atomicCAS(&g_error_word, 0u, site);
  return false;
}

// Sum of one row's cpr partials rr[0 .. cpr) in the fixed order: sequence i (i < 8) adds
// rr[i], rr[i + 8], rr[i + 16], ... from zero; the eight sums combine as
// ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)).  Q lanes share the row (lane q holds the
// sequences q, q + Q, ...); every lane of the group returns the same value, bit for bit, for any Q.
// Loads go out in batches of 48 per lane before the adds that consume them.
template <int Q>
__device__ __forceinline__ float reduce_row(const float* rr, int cpr, int q) {
  constexpr int U = 8 / Q;
  constexpr int R = 48 / U;    // rounds of eight partials per batch
  float a[U];
#pragma unroll
  for (int u = 0; u < U; ++u) a[u] = 0.0f;
  int c0 = 0;
  for (; c0 + 8 * R <= cpr; c0 += 8 * R) {   // full batches
    float v[R][U];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u) v[r][u] = rr[c0 + 8 * r + q + Q * u];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u) a[u] += v[r][u];
  }
  if (c0 < cpr) {                             // the ragged last batch
    float v[R][U];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = c0 + 8 * r + q + Q * u;
        v[r][u] = i < cpr ? rr[i] : 0.0f;
      }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (c0 + 8 * r + q + Q * u < cpr) a[u] += v[r][u];
      }
  }
  if constexpr (Q == 1) {
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  } else {
    // pairs (s0 + s1), (s2 + s3), ...: the partner sequence is one lane away
#pragma unroll
    for (int u = 0; u < U; ++u) a[u] += __shfl_xor_sync(0xffffffffu, a[u], 1);
    if constexpr (Q == 2) {
      return (a[0] + a[1]) + (a[2] + a[3]);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) a[u] += __shfl_xor_sync(0xffffffffu, a[u], 2);
      if constexpr (Q == 4) {
        return a[0] + a[1];
      } else {
        return a[0] + __shfl_xor_sync(0xffffffffu, a[0], 4);
      }
    }
  }
}

template <int FMT, int MB, int MAXL, int MAXG>
__global__ void __launch_bounds__((cons_warps(MB) + 2) * 32, 1)
    w4_persistent_kernel(const __grid_constant__ PParams<MAXL, MAXG> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const PLayout Lo = playout(FMT, p.stages, p.stage_w, p.stage_s, p.red_floats, p.xd_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lo.bar);
  uint64_t* empty = full + kMaxStages;
  uint64_t* rfull = empty + kMaxStages;
  uint64_t* rfree = rfull + kRedBufs;
  // stream gate: 1 while this CTA's consumers compute, 0 while they wait for the previous level
  volatile int* gate = reinterpret_cast<volatile int*>(rfree + kRedBufs);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ncw = p.n_consumer_warps;
  const int n_cons = ncw * 32;
  const int G = (int)gridDim.x;
  const int NS = p.stages;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], ncw);
    }
    for (int i = 0; i < kRedBufs; ++i) {
      mbar_init(&rfull[i], ncw);
      mbar_init(&rfree[i], 1);
    }
    *gate = 1;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == ncw) {
    // ================================================================ producer warp
    if (p.inject_timeout) return;   // test hook: nothing issued, nothing in flight
    const uint64_t pol = policy_evict_first();
    int j = 0;
    bool ok = true;
    for (int L = 0; L < p.nlevels; ++L) {
      const PLevel lv = p.lv[L];
      int g = lv.gemv0;
      for (int t = first_owned(lv.tile0); t < lv.tile0 + lv.ntiles; t += G, ++j) {
        while (t >= p.gm[g].tile0 + p.gm[g].ntiles) ++g;
        const PGemv gm = p.gm[g];
        const int st = j % NS;
        const int round = j / NS;
        // Prefetch of the first NS tiles may overlap the previous kernel in the stream; the
        // bounded waits start only once that kernel is complete.
        if (round == 1 && st == 0) pdl_wait();
        if (lane == 0 && round > 0 && ok) ok = mbar_wait(&empty[st], (round - 1) & 1, 0x201);
        if (lane == 0 && ok) ok = wait_gate(gate, 0x20a);
        if (lane == 0 && NS > kMaxInFlight && j >= kMaxInFlight && ok) {
          const int jd = j - kMaxInFlight;
          ok = mbar_wait(&full[jd % NS], (jd / NS) & 1, 0x209);
        }
        const int r0 = (t - gm.tile0) * gm.rpt;
        const int nrows = min(gm.rpt, gm.N - r0);
        const uint32_t wbytes = (uint32_t)nrows * (uint32_t)(gm.K / 2);
        const uint32_t sbytes = (uint32_t)nrows * (uint32_t)gm.srb;
        const uint32_t sbulk = sbytes & ~15u;
        uint8_t* dst_w = smem + Lo.w + st * p.stage_w;
        uint8_t* dst_s = smem + Lo.s + st * p.stage_s;
        const uint8_t* src_s = reinterpret_cast<const uint8_t*>(gm.scales) + (size_t)r0 * gm.srb;
        if (lane == 0) {
          if (ok) {
            for (uint32_t b = sbulk; b < sbytes; ++b) dst_s[b] = src_s[b];   // sub-16-byte tail
            mbar_arrive_expect_tx(&full[st], wbytes + sbulk);
            bulk_g2s(dst_w, gm.packed + (size_t)r0 * (gm.K / 2), wbytes, &full[st], pol);
            if (sbulk) bulk_g2s(dst_s, src_s, sbulk, &full[st], pol);
          } else {
            mbar_arrive(&full[st]);
          }
        }
        __syncwarp();
      }
    }
    // never leave while bulk copies into this CTA's shared memory may be in flight
    if (lane == 0) {
      for (int k = (j > NS ? j - NS : 0); k < j; ++k) mbar_wait(&full[k % NS], (k / NS) & 1, 0x202);
    }
    return;
  }

  float* red_base = reinterpret_cast<float*>(smem + Lo.red);

  if (warp == ncw + 1) {
    // ================================================================ reducer warp
    pdl_wait();   // counters are touched only after the previous kernel in the stream completed
    int j = 0;
    bool ok = true;
    for (int L = 0; L < p.nlevels; ++L) {
      const PLevel lv = p.lv[L];
      int g = lv.gemv0;
      const int t_end = lv.tile0 + lv.ntiles;
      for (int t = first_owned(lv.tile0); t < t_end; t += G, ++j) {
        while (t >= p.gm[g].tile0 + p.gm[g].ntiles) ++g;
        const PGemv gm = p.gm[g];
        const int b = j % kRedBufs;
        if (ok) ok = mbar_wait(&rfull[b], (j / kRedBufs) & 1, 0x203);
        const int r0 = (t - gm.tile0) * gm.rpt;
        const int nrows = min(gm.rpt, gm.N - r0);
        const float* red = red_base + b * p.red_floats;
        // output o = m * nrows + lr is buffer row o; Q lanes per output
        const int outs = nrows * MB;
        const int Q = red_lanes(outs);
        const int stride = red_stride(gm.cpr, Q);
        const int q = lane & (Q - 1);
        for (int o0 = 0; o0 < outs; o0 += 32 / Q) {
          const int o = o0 + lane / Q;
          const int oc = o < outs ? o : outs - 1;
          const float* rr = red + oc * stride;
          float v;
          switch (Q) {
            case 8: v = reduce_row<8>(rr, gm.cpr, q); break;
            case 4: v = reduce_row<4>(rr, gm.cpr, q); break;
            case 2: v = reduce_row<2>(rr, gm.cpr, q); break;
            default: v = reduce_row<1>(rr, gm.cpr, q); break;
          }
          const int m = oc / nrows;
          if (o < outs && q == 0 && m < p.M) gm.y[(size_t)m * gm.N + r0 + (oc - m * nrows)] = __float2half_rn(v);
        }
        const bool publish = p.counters && t + G >= t_end;   // this CTA's last tile of level L
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&rfree[b]);
          if (publish) {
            if (L + 1 < p.nlevels) *gate = 0;   // before the release: the next level reopens it
            red_release_add(&p.counters[L], 1u);
          }
        }
      }
    }
    // end of the launch: the last CTA to finish resets the counters for the next launch
    asm volatile("bar.sync 2, %0;" ::"r"(n_cons + 32) : "memory");
    if (p.counters && lane == 0) {
      __threadfence();
      const unsigned done = atomicAdd(&p.counters[p.nlevels], 1u);
      if (done == (unsigned)G - 1) {
        for (int L = 0; L <= p.nlevels; ++L) atomicExch(&p.counters[L], 0u);
      }
    }
    return;
  }

  // ================================================================== consumer warps
  const int tid = threadIdx.x;
  const uint32_t lut_lane = smem_u32(smem + Lo.lut) + (uint32_t)lane * 4u;
  if (FMT == 0) build_nf4_lut(reinterpret_cast<uint32_t*>(smem + Lo.lut), p.codebook, tid, n_cons);

  constexpr int kTarget = cons_warps(MB) * 32;
  XSlice<FMT, MB> xs;
  const __half* x_loaded = nullptr;
  int k_loaded = -1;
  int rho = 0, chunk = 0, rps = 1;
  bool active = false;
  int j = 0;
  bool ok = true;
  bool pdl_done = false;
  for (int L = 0; L < p.nlevels; ++L) {
    const PLevel lv = p.lv[L];
    const int t_first = first_owned(lv.tile0);
    const int t_end = lv.tile0 + lv.ntiles;
    if (t_first >= t_end) continue;           // no tile of this level here
    // ---- wait until this level's inputs exist
    if (!pdl_done) {
      pdl_wait();
      pdl_done = true;
    }
    if (L > 0 && p.counters) {
      // every CTA that owns a tile of level L-1 adds one when it has finished them all
      const unsigned owners = (unsigned)min(G, p.lv[L - 1].ntiles);
      if (tid == 0 && ok) ok = wait_counter(&p.counters[L - 1], owners, 0x204);
    }
    // the level's start for all consumers (and the LUT complete at the first level): thread 0's
    // acquire orders every consumer's reads of x after the previous level's writes
    asm volatile("bar.sync 1, %0;" ::"r"(n_cons) : "memory");
    int g = lv.gemv0;
    PGemv gm = p.gm[g];
    for (int t = t_first; t < t_end; t += G, ++j) {
      if (t >= gm.tile0 + gm.ntiles) {
        do { ++g; } while (t >= p.gm[g].tile0 + p.gm[g].ntiles);
        gm = p.gm[g];
      }
      if (gm.x != x_loaded || gm.K != k_loaded) {
        const int cpr = gm.cpr;
        rps = cpr >= kTarget ? 1 : kTarget / cpr;
        rho = tid / cpr;
        chunk = tid - rho * cpr;
        active = rho < rps;
        bool shared_digits = false;
        if constexpr (FMT == 1) {
          if (t == t_first && p.M * cpr * 4 * kXDigitWords <= p.xd_bytes) {
            // INT4: the threads of one row sweep (rho == 0) convert each chunk of x once and share
            // the digits; the level-start barrier above ordered every read of the previous table
            shared_digits = true;
            uint32_t* xd = reinterpret_cast<uint32_t*>(smem + Lo.xd);
            if (rho == 0 && active) {
              load_x_slice<FMT, MB>(xs, gm.x, p.M, gm.K, chunk);
              put_x_digits<MB>(xd, xs, p.M, cpr, chunk);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(n_cons) : "memory");
            if (rho > 0 && active) get_x_digits<MB>(xs, xd, p.M, cpr, chunk);
          }
        }
        if (!shared_digits && active) load_x_slice<FMT, MB>(xs, gm.x, p.M, gm.K, chunk);
        x_loaded = gm.x;
        k_loaded = gm.K;
      }
      if (t == t_first && tid == 0) *gate = 1;
      const int st = j % NS;
      const int b = j % kRedBufs;
      // every lane waits for itself: one instruction per warp, no broadcast round trip
      if (ok) ok = mbar_wait(&full[st], (j / NS) & 1, 0x205);
      if (j >= kRedBufs && ok) ok = mbar_wait(&rfree[b], ((j / kRedBufs) - 1) & 1, 0x206);
      const int r0 = (t - gm.tile0) * gm.rpt;
      const int nrows = min(gm.rpt, gm.N - r0);
      const uint32_t sw = smem_u32(smem + Lo.w + st * p.stage_w);
      const uint32_t ss = smem_u32(smem + Lo.s + st * p.stage_s);
      float* red = red_base + b * p.red_floats;
      const int stride = red_stride(gm.cpr, red_lanes(nrows * MB));
      if (active && ok) {
        const int es = FMT == 0 ? 4 : 2;
        const uint32_t soff = (uint32_t)(((chunk * 32) / gm.bs) * es);
        const uint32_t wrow = (uint32_t)(gm.K / 2);
        int lr = rho;
        for (; lr + rps < nrows; lr += 2 * rps) {   // two rows at once
          const uint4 wv[2] = {lds128(sw + (uint32_t)lr * wrow + chunk * 16),
                               lds128(sw + (uint32_t)(lr + rps) * wrow + chunk * 16)};
          const uint32_t sa[2] = {ss + (uint32_t)(lr * gm.srb) + soff, ss + (uint32_t)((lr + rps) * gm.srb) + soff};
          float part[2][MB];
          chunk_dot<FMT, MB, 2>(part, wv, sa, lut_lane, xs);
#pragma unroll
          for (int m = 0; m < MB; ++m) {
            red[(m * nrows + lr) * stride + chunk] = part[0][m];
            red[(m * nrows + lr + rps) * stride + chunk] = part[1][m];
          }
        }
        if (lr < nrows) {
          const uint4 wv[1] = {lds128(sw + (uint32_t)lr * wrow + chunk * 16)};
          const uint32_t sa[1] = {ss + (uint32_t)(lr * gm.srb) + soff};
          float part[1][MB];
          chunk_dot<FMT, MB, 1>(part, wv, sa, lut_lane, xs);
#pragma unroll
          for (int m = 0; m < MB; ++m) red[(m * nrows + lr) * stride + chunk] = part[0][m];
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[st]);
        mbar_arrive(&rfull[b]);
      }
    }
  }
  asm volatile("bar.sync 2, %0;" ::"r"(n_cons + 32) : "memory");
}

// ====================================================================== host side
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

static int batch_block(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

// Partial-sum floats a tile of nr rows needs.
static int red_floats_for(int MB, int cpr, int nr) {
  const int outs = nr * MB;
  return outs * red_stride(cpr, red_lanes(outs));
}

// Per-GEMV geometry that does not depend on the tiling.
struct GeomG {
  int cpr, srb, align_rows, rpt_max, ncw, rps, red_need;
};

static bool geom(int fmt, int MB, int K, int bs, int stage_target, GeomG& o) {
  o.cpr = K / 32;
  if (o.cpr < 1 || o.cpr > kMaxConsumers) return false;
  const int target = cons_warps(MB) * 32;
  const int rps = o.cpr >= target ? 1 : target / o.cpr;
  o.ncw = (rps * o.cpr + 31) / 32;
  o.srb = (K / bs) * (fmt == 0 ? 4 : 2);
  o.align_rows = 16 / gcd_int(o.srb, 16);       // keeps every tile's scale span 16-byte aligned
  o.rps = rps;
  // about kStageTarget packed bytes, rounded to a whole number of consumer sweeps, within the
  // partial-sum buffer's cap
  const int r = stage_target / (K / 2);
  int sweeps = (r + rps / 2) / rps;
  if (sweeps < 1) sweeps = 1;
  int rows = sweeps * rps;
  while (rows > 1 && red_floats_for(MB, o.cpr, rows) > kRedCapFloats) rows = rows > rps ? rows - rps : rows - 1;
  rows = (rows / o.align_rows) * o.align_rows;
  if (rows < o.align_rows) rows = o.align_rows;
  o.rpt_max = rows;
  o.red_need = 1;
  for (int nr = 1; nr <= rows; ++nr) o.red_need = max(o.red_need, red_floats_for(MB, o.cpr, nr));
  return true;
}

struct Job {
  const uint8_t* packed;
  const void* scales;
  const __half* x;
  __half* y;
  int N, K, bs, level;
};

struct Plan {
  int stage_target, stages, stage_w, stage_s, red_floats, ncw, xd_bytes;
  PLayout L;
};

// Layout of a set of GEMVs at batch block MB (independent of tiling, which never exceeds rpt_max):
// the fixed parts, then as many ring stages (2 ... kMaxStages) as shared memory holds; the stage
// size steps down from kStageTarget until two stages fit.
static bool plan_layout(int fmt, int MB, int M, const Job* jobs, int n, Plan& P) {
  for (P.stage_target = kStageTarget; P.stage_target >= 2048; P.stage_target = P.stage_target * 3 / 4) {
    P.stage_w = 16; P.stage_s = 16; P.red_floats = 1; P.ncw = 1; P.xd_bytes = 0;
    for (int i = 0; i < n; ++i) {
      GeomG gg;
      if (!geom(fmt, MB, jobs[i].K, jobs[i].bs, P.stage_target, gg)) return false;
      P.stage_w = max(P.stage_w, gg.rpt_max * (jobs[i].K / 2));
      P.stage_s = max(P.stage_s, ((gg.rpt_max * gg.srb) + 15) & ~15);
      P.red_floats = max(P.red_floats, gg.red_need);
      P.ncw = max(P.ncw, gg.ncw);
      const int xd = M * gg.cpr * 4 * kXDigitWords;
      if (fmt == 1 && xd <= kXDigitCap) P.xd_bytes = max(P.xd_bytes, xd);
    }
    for (P.stages = kMaxStages; P.stages >= 2; --P.stages) {
      P.L = playout(fmt, P.stages, P.stage_w, P.stage_s, P.red_floats, P.xd_bytes);
      if (P.L.total <= kSmemCap) return true;
    }
  }
  return false;
}

int simt_max_batch(int format, int K, int bs) {
  Job jb{nullptr, nullptr, nullptr, nullptr, 1, K, bs, 0};
  for (int m : {8, 4, 2, 1}) {
    Plan P;
    if (plan_layout(format, m, m, &jb, 1, P)) return m;
  }
  return 0;
}

bool plan_simt(int format, int M, int K, int bs, SimtPlan* out) {
  const int mb = simt_max_batch(format, K, bs);
  if (mb < 1 || M < 1) return false;
  // the widest launch: min(M, mb) rows on the batch block that covers them
  const int mm = M < mb ? M : mb;
  Job jb{nullptr, nullptr, nullptr, nullptr, 1, K, bs, 0};
  Plan P;
  if (!plan_layout(format, batch_block(mm), mm, &jb, 1, P)) return false;
  out->mb = mm;
  out->launches = (M + mb - 1) / mb;
  out->threads = P.ncw * 32 + 64;
  out->smem = P.L.total;
  out->stages = P.stages;
  return true;
}

template <int FMT, int MB, int MAXL, int MAXG>
static cudaError_t launch_persistent(const Job* jobs, int n, int M, const float* codebook, unsigned* counters,
                                     bool pdl, cudaStream_t stream) {
  using P = PParams<MAXL, MAXG>;
  auto kern = w4_persistent_kernel<FMT, MB, MAXL, MAXG>;
  P* pp = new P();   // large parameter block: build on the heap
  P& p = *pp;
  int nlev = 0;
  for (int i = 0; i < n; ++i) nlev = max(nlev, jobs[i].level + 1);
  if (n > MAXG || nlev > MAXL) { delete pp; return cudaErrorNotSupported; }
  Plan plan;
  if (!plan_layout(FMT, MB, M, jobs, n, plan)) {
    delete pp;
    return cudaErrorNotSupported;
  }
  static bool attr_done = false;   // one flag per instance
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
    if (e != cudaSuccess) { delete pp; return e; }
    attr_done = true;
  }
  const int threads = plan.ncw * 32 + 64;
  static int occ_threads = -1, occ_smem = -1, occ_val = 1;
  if (occ_threads != threads || occ_smem != plan.L.total) {
    int v = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, (size_t)plan.L.total);
    if (e != cudaSuccess) { delete pp; return e; }
    occ_threads = threads; occ_smem = plan.L.total; occ_val = v < 1 ? 1 : (v > 2 ? 2 : v);
  }
  const int gmax = device_sm_count() * occ_val;
  p.codebook = codebook;
  p.counters = nlev > 1 ? counters : nullptr;
  if (nlev > 1 && !counters) { delete pp; return cudaErrorInvalidValue; }
  p.nlevels = nlev;
  p.ngemvs = n;
  p.M = M;
  p.inject_timeout = take_fault_injection();
  p.stages = plan.stages; p.stage_w = plan.stage_w; p.stage_s = plan.stage_s; p.red_floats = plan.red_floats;
  p.n_consumer_warps = plan.ncw;
  p.xd_bytes = plan.xd_bytes;
  // tiling, level by level: balanced tiles per CTA, rows per tile within each GEMV's stage budget
  int tile = 0, max_level_tiles = 0;
  for (int Lv = 0, i = 0; Lv < nlev; ++Lv) {
    const int first = i;
    long long rows = 0;
    int rmin = 1 << 30;
    while (i < n && jobs[i].level == Lv) {
      GeomG gg;
      geom(FMT, MB, jobs[i].K, jobs[i].bs, plan.stage_target, gg);
      rows += jobs[i].N;
      rmin = min(rmin, gg.rpt_max);
      ++i;
    }
    p.lv[Lv].gemv0 = first;
    p.lv[Lv].ngemv = i - first;
    p.lv[Lv].tile0 = tile;
    const long long tpc = (rows + (long long)gmax * rmin - 1) / ((long long)gmax * rmin);
    for (int q = first; q < i; ++q) {
      GeomG gg;
      geom(FMT, MB, jobs[q].K, jobs[q].bs, plan.stage_target, gg);
      int rpt = (int)((rows + (long long)gmax * tpc - 1) / ((long long)gmax * tpc));
      if (rpt > gg.rps) rpt = ((rpt + gg.rps - 1) / gg.rps) * gg.rps;   // whole sweeps when it can
      rpt = ((rpt + gg.align_rows - 1) / gg.align_rows) * gg.align_rows;
      rpt = min(rpt, gg.rpt_max);
      PGemv& g = p.gm[q];
      g.packed = jobs[q].packed; g.scales = jobs[q].scales; g.x = jobs[q].x; g.y = jobs[q].y;
      g.N = jobs[q].N; g.K = jobs[q].K; g.bs = jobs[q].bs; g.rpt = rpt;
      g.tile0 = tile; g.ntiles = (g.N + rpt - 1) / rpt; g.srb = gg.srb; g.cpr = gg.cpr;
      tile += g.ntiles;
    }
    p.lv[Lv].ntiles = tile - p.lv[Lv].tile0;
    max_level_tiles = max(max_level_tiles, p.lv[Lv].ntiles);
  }
  const int grid = nlev > 1 ? gmax : min(gmax, max_level_tiles);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)plan.L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  delete pp;
  return e;
}

template <int MAXL, int MAXG>
static cudaError_t dispatch(int fmt, int MB, const Job* jobs, int n, int M, const float* codebook, unsigned* counters,
                            bool pdl, cudaStream_t s) {
  if (fmt == 0) {
    switch (MB) {
      case 1: return launch_persistent<0, 1, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
      case 2: return launch_persistent<0, 2, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
      case 4: return launch_persistent<0, 4, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
      default: return launch_persistent<0, 8, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
    }
  }
  switch (MB) {
    case 1: return launch_persistent<1, 1, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
    case 2: return launch_persistent<1, 2, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
    case 4: return launch_persistent<1, 4, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
    default: return launch_persistent<1, 8, MAXL, MAXG>(jobs, n, M, codebook, counters, pdl, s);
  }
}

cudaError_t launch_gemv_simt(int format, const uint8_t* packed, const void* scales, const float* codebook,
                             const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                             cudaStream_t stream) {
  if (M < 1 || M > 8) return cudaErrorNotSupported;
  Job jb{packed, scales, x, y, N, K, bs, 0};
  return dispatch<1, 1>(format, batch_block(M), &jb, 1, M, codebook, nullptr, pdl, stream);
}

cudaError_t launch_step_simt(int format, const StepJob* jobs, int n, int M, const float* codebook, unsigned* counters,
                             bool pdl, cudaStream_t stream) {
  if (M < 1 || M > 8 || n < 1 || n > kStepMaxGemvs) return cudaErrorNotSupported;
  Job js[kStepMaxGemvs];
  for (int i = 0; i < n; ++i) {
    js[i] = Job{jobs[i].packed, jobs[i].scales, jobs[i].x, jobs[i].y, jobs[i].N, jobs[i].K, jobs[i].bs, jobs[i].level};
  }
  return dispatch<kStepMaxGemvs, kStepMaxGemvs>(format, batch_block(M), js, n, M, codebook, counters, pdl, stream);
}

// ---------------------------------------------------------------------------------------------
// Counters for w4_gemv_levels_noalloc: a fixed array inside the library, for callers that cannot
// allocate device memory.  In host code the name g_noalloc_counters is only a stand-in for the
// device object; its device address is looked up once per device and cached.
constexpr int kNoAllocMaxLevels = 256;
constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned int g_noalloc_counters[kNoAllocMaxLevels + 1];

static cudaError_t noalloc_counters(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  static std::mutex mu;
  static unsigned* addr[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_counters);   // with this device current
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<unsigned*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

int noalloc_max_levels() { return kNoAllocMaxLevels; }

cudaError_t launch_step_simt_noalloc(int format, const StepJob* jobs, int n, int M, const float* codebook,
                                     int nlevels, cudaStream_t stream) {
  if (nlevels < 1 || nlevels > kNoAllocMaxLevels) return cudaErrorInvalidValue;
  unsigned* counters = nullptr;
  cudaError_t e = noalloc_counters(&counters);
  if (e != cudaSuccess) return e;
  // the array keeps the previous call's contents: start from zero
  e = cudaMemsetAsync(counters, 0, sizeof(unsigned) * (size_t)(nlevels + 1), stream);
  if (e != cudaSuccess) return e;
  return launch_step_simt(format, jobs, n, M, codebook, counters, true, stream);
}

unsigned int read_clear_error_persist() { return read_clear_error_word_here(); }

}  // namespace w4
