// w4_persist.cu -- fused 4-bit dequant-GEMV for batches 1 ... 8 (sm_103a): one persistent,
// warp-specialised kernel for a single GEMV or for every GEMV of a decode step.
//
// Computes y[m][n] = sum_k w_hat[n][k] * x[m][k] with w_hat decoded on chip, FP32 accumulation and
// an FP16 result; no dequantised matrix ever reaches DRAM ("LLM Quantization on RTX 4060: Where
// 4-bit Decode Falls Behind FP16", sections "Fused Kernel: Moving Dequantization On-Chip" and
// "Kernel Implementation").
//
// Work: each GEMV is cut into tiles of whole rows.  GEMVs are grouped into levels; a level's GEMVs
// are independent of each other (the projections of one decode layer that read the same
// activation: q, k, v / o / gate, up / down).  A level's x is read only after every tile of the
// previous level is complete, which models the decode step's data dependencies ("Do Quantization
// and Sparsity make LLM Inference Faster ?", section "What we did": the 197 GEMVs of one step).
// Level 0 waits for the previous kernel in the stream (programmatic dependent launch); later levels
// wait on counters in global memory.  Tile t of a level goes to CTA t mod gridDim.x; the grid is
// one CTA per SM, all co-resident.
//
// The arithmetic runs on the tensor cores through warp-level mma.sync.m16n8k16 (FP16 x FP16 ->
// FP32), with the weights as the A operand and x (batch rows 0 ... 7; columns at or above the batch
// are computed from the last batch row and never stored) as B:
//   * a warp's unit of work is 16 rows x 128 k of one tile (a "span"): per 64-k block (32-k block
//     when the scale block is 32) lane (g, t) = (lane / 4, lane % 4) reads the 8 (4) consecutive
//     packed bytes 8t ... 8t + 7 of the rows its MMA rows g and g + 8 stand for (tile rows 2g and
//     2g + 1 of the row group with 64-k blocks, g and g + 8 with 32-k blocks, the pairing that keeps
//     the swizzled loads conflict-free); each byte is one A-fragment register, two
//     consecutive k of one row, decoded by one shared-memory lookup in a byte-pair table (NF4 code
//     values, q - 8 for INT4, E2M1 values for FP4, all exact in FP16 except the NF4 code values,
//     which are rounded to FP16).  At batch 1 the table is 64 KB (entries 256 bytes apart, so one
//     byte permute forms a lookup's offset from the packed byte and the lane, and the table's
//     address folds into the load) and its free halves hold the partial sums; above batch 1 it is
//     32 KB (one shift-add per lookup).  K is permuted identically in A and B, so the B fragment is
//     the lane's own x elements, loaded in natural order;
//   * the MMAs of one scale block start from zero, and the block's scale (FP32 absmax for NF4,
//     FP16 scale for INT4 and FP4) multiplies the result into the unit's FP32 accumulators;
//   * each unit leaves one FP32 partial per (batch row, weight row, span) in shared memory, and the
//     reducer warp sums a row's spans in an order that depends only on K (eight interleaved
//     sequences, then a fixed tree), so a row gets the same bits whatever the tiling.
// Roles in a CTA:
//   * producer warp: copies each tile into a shared-memory ring with one 2-D TMA tensor copy per
//     256-k box (128 bytes x the tile's rows, 128-byte swizzled: the 16-byte chunk c of tile row r
//     lands at chunk c ^ (r & 7), so the fragment loads of a warp hit distinct banks) and its scales
//     with one 1-D bulk copy, completion on the stage's mbarrier.  Weights never depend on other
//     GEMVs, so it runs ahead across level boundaries.  Copies are issued only while the CTA's
//     consumers compute (a stream gate opened once a level starts and closed before the stage of
//     the CTA's last tile of the level is released), because data arriving at the SM while a
//     level's completion is published and the next level waits slows that release and its polls.
//     The consumers open the gate before they wait for a level's first tile, so a tile held back
//     at a level's end is issued as soon as the level starts;
//   * 14 consumer warps (16 warps in all, so each thread may hold 128 registers): each takes a
//     contiguous chunk of the tile's units in span-major order (consecutive units of a warp share a
//     span, so its x stays in registers while the row group advances); chunk sizes differ by at
//     most one and the warps that take the larger ones rotate from tile to tile;
//   * reducer warp: sums each row's partials, writes y, and after the CTA's last tile of a level
//     publishes completion with one release, before it reads any table entry of the next tile
//     (whether a tile ends the CTA's part of a level is known from the cursor alone).
// Every wait is bounded in wall-clock time; a lost wait is recorded in the device error word and
// the kernel runs to its end without further waiting.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4.h"
#include "w4_common.cuh"
#include "w4_decode.cuh"
#include "w4_internal.h"
#include "w4_mma_unit.cuh"

namespace w4 {

constexpr int kMaxStages = 8;
constexpr int kMaxInFlight = 3;        // tile copies outstanding per CTA
constexpr int kConsumerWarps = 14;
constexpr int kThreads = (kConsumerWarps + 2) * 32;   // consumers, producer, reducer
constexpr int kStageTarget = 65536;    // packed bytes per stage (about); smaller when the ring won't fit
constexpr int kRedBufs = 2;            // partial-sum buffers: the reducer may lag one tile
constexpr int kRedCapFloats = 12288;   // largest partial-sum buffer (floats)
constexpr int kSmemCap = 227 * 1024;
constexpr int kMaxRowsPerTile = 256;  // TMA box rows

__host__ __device__ constexpr int span_count(int K) { return (K + kSpanK - 1) / kSpanK; }
__host__ __device__ constexpr int box_count(int K) { return (K + kBoxK - 1) / kBoxK; }
// Shared-memory bytes of one TMA box of a tile of `rows` rows: whole 1 KB swizzle atoms (8 rows of
// 128 bytes; the 128-byte swizzle wants 1 KB aligned boxes).
__host__ __device__ constexpr int span_slot(int rows) { return ((rows + 7) / 8) * 1024; }
// A stage: the boxes of a tile, then 1 KB that the last row group may read past the last box (its
// rows beyond the tile are never used).
__host__ __device__ constexpr int stage_bytes(int nbox, int rows) { return nbox * span_slot(rows) + 1024; }
// Floats per (batch row, weight row) in a partial-sum buffer: at least the span count and 4 more
// than a multiple of 8, so rows are 16-byte aligned and the reducer's 16-byte loads of eight
// consecutive outputs hit distinct banks.
__host__ __device__ constexpr int part_stride(int C) { return C + ((4 - C) & 7); }
// Floats a partial-sum buffer holds past its last row: the reducer reads whole groups of eight
// spans.
constexpr int kRedSlackFloats = 8;

struct PGemv {
  const uint8_t* packed;
  const void* scales;
  const __half* x;
  __half* y;
  const CUtensorMap* tmap; // packed [N][K/2], box 128 bytes x rpt rows (device memory; null: map1)
  int N, K, bs, rpt;       // rpt: rows per tile
  int tile0, ntiles, srb;  // global tile range; scale bytes per row
  int nspan, nbox, slot, cp;  // spans (128 k) and TMA boxes (256 k) per row; shared bytes per box;
                              // partial stride (floats)
  int pad_[3];
};
static_assert(sizeof(PGemv) % 16 == 0, "PGemv is read as 16-byte vectors");

struct PLevel {
  int gemv0;
  int wait;                // releases this level waits for: the CTAs owning tiles of the level before
  int tile0, ntiles;
};

// Launch parameters.  A single-GEMV launch carries its level, GEMV and tensor map here; a
// multi-GEMV launch reads them from tables in device memory (written once by the host), because a
// parameter block large enough for a decode step does not stay in the constant cache and every
// tile would pay for that.
struct PParams {
  CUtensorMap map1;        // the tensor map of a single-GEMV launch
  const float* codebook;   // NF4 code book (format 0)
  unsigned int* counters;  // [nlevels + 1] when nlevels > 1, else null
  const PLevel* lvt;       // device tables of a multi-GEMV launch (null: lv1 and gm1)
  const PGemv* gmt;
  int fmt;                 // 0 NF4 (FP32 absmax), 1 INT4 (FP16 scale), 2 FP4 E2M1 (FP16 scale)
  int nlevels, ngemvs, M, inject_timeout;
  int stages, stage_w, stage_s, red_floats;
  PLevel lv1;
  PGemv gm1;
};

template <class T>
__device__ __forceinline__ T ldg_struct(const T* q) {
  T v;
  const uint4* src = reinterpret_cast<const uint4*>(q);
  uint4* dst = reinterpret_cast<uint4*>(&v);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(T) / 16); ++i) dst[i] = __ldg(src + i);
  return v;
}
__device__ __forceinline__ PLevel level_at(const PParams& p, int L) { return p.lvt ? ldg_struct(p.lvt + L) : p.lv1; }
__device__ __forceinline__ PGemv gemv_at(const PParams& p, int g) { return p.gmt ? ldg_struct(p.gmt + g) : p.gm1; }

struct PLayout {
  int lut, w, s, red, bar, total;
};

// The 64 KB table's gaps (entry b's bytes 128 ... 255) hold the two partial-sum buffers at batch 1:
// gaps 0 ... 127 the first, 128 ... 255 the second.
constexpr int kGapOffset = 128;
constexpr int kGapsPerBuf = 128;
constexpr int kGapBufBytes = kGapsPerBuf * 256;
__host__ __device__ constexpr int gaps_per_output(int nspan) { return (nspan + 31) >> 5; }

// wide: the 64 KB table, the partial sums in its gaps (red_floats unused).
__host__ __device__ inline PLayout playout(int stages, int stage_w, int stage_s, int red_floats, bool wide) {
  PLayout L;
  int off = 0;
  L.lut = off;
  off += wide ? kLutWideBytes : kLutBytes;   // 32 or 64 KB: the ring starts 1 KB aligned
  L.w = off;
  off += stages * stage_w;
  L.s = off;
  off += stages * stage_s;
  off = (off + 15) & ~15;
  L.red = off;
  if (!wide) off += kRedBufs * red_floats * 4;
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

// Adds v with release semantics at GPU scope: every write ordered before it (this thread's, and
// its warp's through a preceding __syncwarp) is visible to a thread that acquires the new value.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
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

// 2-D TMA tensor copy global -> shared (box at coordinates c0 = byte column, c1 = row); completion
// adds the box's bytes to `bar`.  dst: 1 KB aligned shared address.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                       uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}


// The tiles of one CTA, in order across levels: level, GEMV (index and descriptor) and global tile
// index, with the end tiles of the current level and GEMV kept, so that a step reads the tables
// only when it moves on and "is this the CTA's last tile of its level" needs no table read.
struct TileCursor {
  int L, g, t, lend, gend, wait;
  PGemv gm;
  __device__ __forceinline__ void start(const PParams& p) {
    L = 0;
    seek(p);
  }
  __device__ __forceinline__ void find_gemv(const PParams& p) {
    for (;;) {
      gm = gemv_at(p, g);
      gend = gm.tile0 + gm.ntiles;
      if (t < gend) break;
      ++g;
    }
  }
  // this is the CTA's last tile of level L (the next one, if any, belongs to a later level)
  __device__ __forceinline__ bool level_last() const { return t + (int)gridDim.x >= lend; }
  // from level L on: this CTA's first tile of the first level that has one
  __device__ __forceinline__ void seek(const PParams& p) {
    while (L < p.nlevels) {
      const PLevel lv = level_at(p, L);
      t = first_owned(lv.tile0);
      lend = lv.tile0 + lv.ntiles;
      wait = lv.wait;
      if (t < lend) {
        g = lv.gemv0;
        find_gemv(p);
        return;
      }
      ++L;
    }
  }
  __device__ __forceinline__ bool valid(const PParams& p) const { return L < p.nlevels; }
  __device__ __forceinline__ void next(const PParams& p) {
    t += (int)gridDim.x;
    if (t >= lend) {
      ++L;
      seek(p);
      return;
    }
    if (t >= gend) {
      ++g;
      find_gemv(p);
    }
  }
};

// The reducer's work for one tile with more outputs than lanes: each lane sums R outputs
// o = base + lane + 32 r at once.
template <int R, class Part>
__device__ __forceinline__ void reduce_tile_batched(const Part& P, const PGemv& gm, int outs, int nrows, int r0,
                                                    int lane) {
  for (int base = 0; base < outs; base += 32 * R) {
    int oo[R];
#pragma unroll
    for (int r = 0; r < R; ++r) oo[r] = min(base + lane + 32 * r, outs - 1);
    float v[R];
    sum_spans_batch<R>(v, P, oo, gm.nspan);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int o = base + lane + 32 * r;
      if (o < outs) {
        const int m = o / nrows;
        gm.y[(size_t)m * gm.N + r0 + (o - m * nrows)] = __float2half_rn(v[r]);
      }
    }
  }
}

// The reducer's work for one tile: each output o = m * nrows + r (batch row m, tile row r) summed
// over its spans by Q lanes, written to y as FP16.
template <int Q, class Part>
__device__ __forceinline__ void reduce_tile(const Part& P, const PGemv& gm, int outs, int nrows, int r0,
                                            int lane) {
  for (int base = 0; base < outs; base += 32 / Q) {
    const int o = base + lane / Q;
    const float v = sum_spans<Q>(P, min(o, outs - 1), gm.nspan, lane % Q);
    if (o < outs && lane % Q == 0) {
      const int m = o / nrows;
      gm.y[(size_t)m * gm.N + r0 + (o - m * nrows)] = __float2half_rn(v);
    }
  }
}

// As many lanes per output (1, 2, 4 or 8) as make one pass over the tile's outputs.
template <class Part>
__device__ __forceinline__ void reduce_tile_any(const Part& P, const PGemv& gm, int outs, int nrows, int r0,
                                                int lane) {
  if (outs <= 4) reduce_tile<8>(P, gm, outs, nrows, r0, lane);
  else if (outs <= 8) reduce_tile<4>(P, gm, outs, nrows, r0, lane);
  else if (outs <= 16) reduce_tile<2>(P, gm, outs, nrows, r0, lane);
  else reduce_tile_batched<4>(P, gm, outs, nrows, r0, lane);
}

// NSCF: the number of block scales per full span when every GEMV of the launch has the same block
// size (1, 2 or 4), compiled in; 0 when they differ (the general unit serves every span).
// WIDE: the 64 KB byte-pair table, with the partial sums in its gaps (batch 1 only).
template <int KB, bool SC32, int NSCF, bool WIDE>
__global__ void __launch_bounds__(kThreads, 1) w4_persistent_kernel(const __grid_constant__ PParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const PLayout Lo = playout(p.stages, p.stage_w, p.stage_s, p.red_floats, WIDE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lo.bar);
  uint64_t* empty = full + kMaxStages;
  uint64_t* rfull = empty + kMaxStages;
  uint64_t* rfree = rfull + kRedBufs;
  // stream gate: 1 while this CTA's consumers compute, 0 while they wait for the previous level
  volatile int* gate = reinterpret_cast<volatile int*>(rfree + kRedBufs);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_cons = kConsumerWarps * 32;
  const int G = (int)gridDim.x;
  const int NS = p.stages;
  if (WIDE && p.M != 1) {   // the gaps hold batch 1's partials only (the host never launches this)
    if (threadIdx.x == 0) atomicCAS(&g_error_word, 0u, 0x20bu);
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kRedBufs; ++i) {
      mbar_init(&rfull[i], kConsumerWarps);
      mbar_init(&rfree[i], 1);
    }
    *gate = 1;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ================================================================ producer warp
    if (p.inject_timeout) return;   // test hook: nothing issued, nothing in flight
    const uint64_t pol = policy_evict_first();
    TileCursor cur;
    cur.start(p);
    int j = 0;
    bool ok = true;
    for (; cur.valid(p); cur.next(p), ++j) {
      const PGemv& gm = cur.gm;
      const int st = j % NS;
      const int round = j / NS;
      // Copies of the first NS tiles may overlap the previous kernel in the stream; the bounded
      // waits start only once that kernel is complete.
      if (round == 1 && st == 0) pdl_wait();
      if (lane == 0 && round > 0 && ok) ok = mbar_wait(&empty[st], (round - 1) & 1, 0x201);
      if (lane == 0 && ok) ok = wait_gate(gate, 0x20a);
      if (lane == 0 && NS > kMaxInFlight && j >= kMaxInFlight && ok) {
        const int jd = j - kMaxInFlight;
        ok = mbar_wait(&full[jd % NS], (jd / NS) & 1, 0x209);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      const int r0 = (cur.t - gm.tile0) * gm.rpt;
      const int nrows = min(gm.rpt, gm.N - r0);
      const uint32_t sbytes = (uint32_t)nrows * (uint32_t)gm.srb;
      const uint32_t sbulk = sbytes & ~15u;
      const uint32_t dst_w = smem_u32(smem + Lo.w + st * p.stage_w);
      uint8_t* dst_s = smem + Lo.s + st * p.stage_s;
      const uint8_t* src_s = reinterpret_cast<const uint8_t*>(gm.scales) + (size_t)r0 * gm.srb;
      const CUtensorMap* tm = gm.tmap ? gm.tmap : &p.map1;
      if (lane == 0) {
        if (ok) {
          for (uint32_t b = sbulk; b < sbytes; ++b) dst_s[b] = src_s[b];   // sub-16-byte tail
          // every box carries rpt rows (zeros past the matrix)
          mbar_arrive_expect_tx(&full[st], (uint32_t)gm.nbox * (uint32_t)gm.rpt * 128u + sbulk);
        } else {
          mbar_arrive(&full[st]);
        }
      }
      __syncwarp();
      if (ok) {
        for (int c = lane; c < gm.nbox; c += 32)
          tma_2d(dst_w + (uint32_t)(c * gm.slot), tm, c * (kBoxK / 2), r0, &full[st], pol);
        if (lane == 31 && sbulk) bulk_g2s(dst_s, src_s, sbulk, &full[st], pol);
      }
      __syncwarp();
    }
    // never leave while bulk copies into this CTA's shared memory may be in flight
    if (lane == 0) {
      for (int k = (j > NS ? j - NS : 0); k < j; ++k) mbar_wait(&full[k % NS], (k / NS) & 1, 0x202);
    }
    return;
  }

  float* red_base = reinterpret_cast<float*>(smem + Lo.red);

  if (warp == kConsumerWarps + 1) {
    // ================================================================ reducer warp
    pdl_wait();   // counters are touched only after the previous kernel in the stream completed
    TileCursor cur;
    cur.start(p);
    int j = 0;
    bool ok = true;
    for (; cur.valid(p); ++j) {
      const int L = cur.L;
      const PGemv& gm = cur.gm;
      const int t = cur.t;
      const int b = j % kRedBufs;
      if (ok) ok = mbar_wait(&rfull[b], (j / kRedBufs) & 1, 0x203);
      const int r0 = (t - gm.tile0) * gm.rpt;
      const int nrows = min(gm.rpt, gm.N - r0);
      // output o = m * nrows + r (batch row m, tile row r)
      const int outs = nrows * p.M;
      if (WIDE) {
        const PartGaps P{smem + Lo.lut + kGapOffset + b * kGapBufBytes, gaps_per_output(gm.nspan)};
        reduce_tile_any(P, gm, outs, nrows, r0, lane);
      } else {
        const PartDense P{red_base + b * p.red_floats, gm.cp};
        reduce_tile_any(P, gm, outs, nrows, r0, lane);
      }
      // the CTA's last tile of level L: publish before the cursor reads the next tile's tables
      const bool publish = p.counters && cur.level_last();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&rfree[b]);
        if (publish) red_release_add(&p.counters[L], 1u);
      }
      cur.next(p);
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
  build_lut(reinterpret_cast<uint32_t*>(smem + Lo.lut), p.fmt, p.codebook, tid, n_cons, WIDE);
  asm volatile("bar.sync 1, %0;" ::"r"(n_cons) : "memory");   // the table is read before the first level
  // 32 KB table: the lane's entry 0; 64 KB table: the table (the lane enters through the permute)
  const uint32_t lut_lane = smem_u32(smem + Lo.lut) + (WIDE ? 0u : (uint32_t)lane * 4u);
  constexpr int RUN = KB / 8;
  constexpr int NKB = kSpanK / KB;
  const int g = lane >> 2, tq = lane & 3;
  // this lane's byte offset of k block j of a span within a swizzled 128-byte box row: bytes
  // 64 h + (KB/2) j + RUN t ... (h: which half of the box the span is) of tile row r sit in 16-byte
  // chunk (64 h + (KB/2) j + RUN t) / 16 ^ (r & 7), i.e. the offset for h = 0 XOR (h << 6); the rows
  // of MMA rows g and g + 8 have r & 7 = 2g & 7, 2g + 1 & 7 (64-k blocks) or g, g (32-k blocks)
  uint32_t off0[NKB], off1[NKB];
  {
    const int x0 = KB == 64 ? (2 * g) & 7 : g, x1 = KB == 64 ? (2 * g + 1) & 7 : g;
#pragma unroll
    for (int jj = 0; jj < NKB; ++jj) {
      const int byte = (KB / 2) * jj + RUN * tq;
      off0[jj] = (uint32_t)((((byte >> 4) ^ x0) << 4) | (byte & 15));
      off1[jj] = (uint32_t)((((byte >> 4) ^ x1) << 4) | (byte & 15));
    }
  }
  constexpr int DSUB = KB == 64 ? 1 : 8;   // tile row of MMA row g + 8 minus that of MMA row g
  const int rsub = KB == 64 ? 2 * g : g;   // tile row of MMA row g within its row group
  int j = 0;
  int st = 0;               // ring stage of tile j and the parity of its current round
  uint32_t sph = 0;
  int wrot = 0;             // the warp that takes the first chunk of the next tile
  bool ok = true;
  bool pdl_done = false;
  TileCursor cur;
  cur.start(p);
  int Lcur = -1;
  for (; cur.valid(p); cur.next(p), ++j) {
    const int L = cur.L;
    const PGemv& gm = cur.gm;
    const int b = j & 1;
    const int r0 = (cur.t - gm.tile0) * gm.rpt;
    const int nrows = min(gm.rpt, gm.N - r0);
    const int rgs = (nrows + 15) >> 4;
    const int units = rgs * gm.nspan;
    const uint32_t tile_s = smem_u32(smem + Lo.w + st * p.stage_w);
    const uint32_t stile_s = smem_u32(smem + Lo.s + st * p.stage_s);
    const uint32_t red_s = smem_u32(red_base + b * p.red_floats);
    // x of batch row g (the last batch row in lanes above the batch: those B columns are never
    // stored)
    const uint8_t* xrow = reinterpret_cast<const uint8_t*>(gm.x + (size_t)min(g, p.M - 1) * gm.K) + (KB / 2) * tq;
    // this warp's units: a contiguous chunk of the tile's units in span-major order
    // u = c * rgs + rg (c: span, rg: row group), so that consecutive units share x; chunk sizes
    // differ by at most one, and the warps that take the larger ones rotate from tile to tile
    int wq = warp - wrot;
    if (wq < 0) wq += kConsumerWarps;
    const int uq = units / kConsumerWarps, ur = units - uq * kConsumerWarps;
    const int u_begin = wq * uq + min(wq, ur);
    int left = uq + (wq < ur ? 1 : 0);
    wrot += ur;
    if (wrot >= kConsumerWarps) wrot -= kConsumerWarps;
    const bool is_level_end = cur.level_last() && L + 1 < p.nlevels;
    if (L != Lcur) {
      // ---- this CTA's first tile of the level: wait until this level's inputs exist
      if (!pdl_done) {
        pdl_wait();
        pdl_done = true;
      }
      if (L > 0 && p.counters) {
        // every CTA that owns a tile of level L-1 adds one when it has finished them all
        if (tid == 0 && ok) ok = wait_counter(&p.counters[L - 1], (unsigned)cur.wait, 0x204);
      }
      // the level's start for all consumers: thread 0's acquire orders every consumer's reads of
      // x after the previous level's writes
      asm volatile("bar.sync 1, %0;" ::"r"(n_cons) : "memory");
      if (tid == 0) *gate = 1;
      Lcur = L;
    }
    // every lane waits for itself: one instruction per warp, no broadcast round trip
    if (ok) ok = mbar_wait(&full[st], sph, 0x205);
    if (j >= kRedBufs && ok) ok = mbar_wait(&rfree[b], ((j >> 1) - 1) & 1, 0x206);
    if (ok && left > 0) {
      const bool full_last = (gm.K % kSpanK) == 0;   // every span full, scale runs aligned
      const int lgbs = 31 - __clz(gm.bs);
      const int sshift = 31 - __clz(gm.bs / KB);
      // first unit of the chunk: u_begin / rgs, exact in FP32 (u_begin < 2^11, rgs <= 16)
      int c = (int)(((float)u_begin + 0.5f) * __frcp_rn((float)rgs));
      int rg = u_begin - c * rgs;
      if (rg < 0) { --c; rg += rgs; }        // never taken (the quotient is exact); keeps 0 <= rg < rgs
      if (rg >= rgs) { ++c; rg -= rgs; }
      // partial-sum rows of batch rows 2t and 2t + 1 (stored only where those rows exist)
      const bool m0 = 2 * tq < p.M, m1 = 2 * tq + 1 < p.M;
      const uint32_t pm0 = red_s + (uint32_t)(2 * tq * nrows * gm.cp) * 4u;
      const uint32_t pm1 = pm0 + (uint32_t)(nrows * gm.cp) * 4u;
      const uint32_t pdsub = (uint32_t)(DSUB * gm.cp) * 4u;
      // gaps (batch 1): output r's span c at gap r * hpo + c / 32, word (c + 4 (r & 7)) mod 32
      const int hpo = gaps_per_output(gm.nspan);
      const uint32_t gap_s = smem_u32(smem + Lo.lut + kGapOffset + b * kGapBufBytes);
      const int rot_a = 4 * (rsub & 7), rot_b = 4 * ((rsub + DSUB) & 7);   // r & 7 of rows ra, rb
      // the chunk's units; FULL: every span full, each row's span scales one aligned vector
      // (NSCF = max(1, 128 / bs)), decided once per tile
      auto run_chunk = [&](auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
        constexpr int NSC = FULL ? NSCF : 0;
        while (left > 0) {
          // ---- span c: x, its box and half, its scale column
          uint32_t xr[NKB][KB / 8];
          const uint8_t* xg = xrow + c * (kSpanK * 2);
          const int nkb = min(kSpanK, gm.K - c * kSpanK) / KB;
          const int sidx0 = (c * kSpanK) >> lgbs;
          load_span_x<KB, FULL>(xr, xg, nkb);
          const uint32_t bc = tile_s + (uint32_t)((c >> 1) * gm.slot + rsub * 128) + ((uint32_t)(c & 1) << 6);
          const uint32_t sc = stile_s + (uint32_t)(FULL ? sidx0 * (SC32 ? 4 : 2) : 0);
          const uint32_t ga = gap_s + (uint32_t)(((c >> 5) << 8) + ((((c & 31) + rot_a) & 31) << 2));
          const uint32_t gb = gap_s + (uint32_t)(((c >> 5) << 8) + ((((c & 31) + rot_b) & 31) << 2)) +
                              (uint32_t)(DSUB * hpo * 256);
          const int cnt = min(left, rgs - rg);
          for (int i = 0; i < cnt; ++i, ++rg) {
            const int ra = rg * 16 + rsub, rb = ra + DSUB;
            const uint32_t b0 = bc + (uint32_t)rg * 2048u, b1 = b0 + DSUB * 128u;
            const uint32_t s0a = sc + (uint32_t)(min(ra, nrows - 1) * gm.srb);
            const uint32_t s1a = sc + (uint32_t)(min(rb, nrows - 1) * gm.srb);
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_unit<KB, SC32, NSC, WIDE>(acc, b0, b1, off0, off1, s0a, s1a, xr, FULL ? 0 : sidx0, sshift, nkb,
                                          lut_lane, lane);
            const bool va = ra < nrows, vb = rb < nrows;
            if (WIDE) {
              // batch 1: batch row 0 of weight rows ra and rb (lanes t = 0)
              const uint32_t go = (uint32_t)(ra * hpo) << 8;
              sts_f32_if(ga + go, acc[0], m0 && va);
              sts_f32_if(gb + go, acc[2], m0 && vb);
            } else {
              // partials: batch rows 2t, 2t + 1 of weight rows ra and rb, at red[(m * nrows + r) * cp + c]
              const uint32_t o = (uint32_t)(ra * gm.cp + c) * 4u;
              sts_f32_if(pm0 + o, acc[0], m0 && va);
              sts_f32_if(pm0 + o + pdsub, acc[2], m0 && vb);
              sts_f32_if(pm1 + o, acc[1], m1 && va);
              sts_f32_if(pm1 + o + pdsub, acc[3], m1 && vb);
            }
          }
          left -= cnt;
          rg = 0;
          ++c;
        }
      };
      if constexpr (NSCF > 0) {
        if (full_last) run_chunk(std::true_type{});
        else run_chunk(std::false_type{});
      } else {
        run_chunk(std::false_type{});
      }
    }
    __syncwarp();
    if (lane == 0) {
      // the CTA's last tile of a level: close the stream gate before this stage is released, so
      // that no copy is issued (and in flight) while the level's completion is published and the
      // next level waits; the next level's start reopens it
      if (p.counters && is_level_end) *gate = 0;
      mbar_arrive(&empty[st]);
      mbar_arrive(&rfull[b]);
    }
    if (++st == NS) {
      st = 0;
      sph ^= 1u;
    }
  }
  asm volatile("bar.sync 2, %0;" ::"r"(n_cons + 32) : "memory");
}

// ====================================================================== host side
// Per-device values the host side looks up once (SM counts; the kernels' attribute set-up and
// occupancy): a fixed table indexed by device, guarded by one mutex.
constexpr int kMaxDevices = 64;

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int device_sm_count() {
  static std::mutex mu;
  static int sms[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (sms[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 1;
  }
  return sms[dev];
}

static int gcd_int(int a, int b) {
  while (b) { int t = a % b; a = b; b = t; }
  return a;
}

// Per-GEMV geometry: scale bytes per row, the row count that keeps every tile's scale span 16-byte
// aligned, the largest tile, spans per row, partial stride and partial floats.
struct GeomG {
  int srb, align_rows, rpt_max, nspan, nbox, cp, red_need;
};

static int kb_of(int bs) { return bs >= 64 ? 64 : 32; }

static bool shape_ok(int K, int bs) { return K >= 32 && K % 32 == 0 && K <= W4_MAX_K && bs >= 32 && K % bs == 0; }

struct Job {
  const uint8_t* packed;
  const void* scales;
  const __half* x;
  __half* y;
  int N, K, bs, level;
};

// Rows per tile and its constraints for one GEMV at a stage budget (bytes of packed data).  wide:
// the partial sums live in the 64 KB table's gaps (batch 1), which bounds the rows of a tile.
static void tile_rows(int fmt, int M, int K, int bs, int stage_target, bool wide, GeomG& o) {
  o.nspan = span_count(K);
  o.nbox = box_count(K);
  o.cp = part_stride(o.nspan);
  o.srb = (K / bs) * (fmt == 0 ? 4 : 2);
  o.align_rows = 16 / gcd_int(o.srb, 16);       // keeps every tile's scale span 16-byte aligned
  int rows = stage_target / (o.nbox * 128);
  if (rows > 16) rows &= ~15;                   // whole MMA row groups when the tile has several
  rows = max(1, min(rows, kMaxRowsPerTile));
  while (rows > 1 && rows * M * o.cp > kRedCapFloats) rows = rows > 16 ? rows - 16 : rows - 1;
  if (wide) {
    const int cap = kGapsPerBuf / gaps_per_output(o.nspan);   // outputs per gap buffer (M = 1)
    while (rows > 1 && rows > cap) rows = rows > 16 ? rows - 16 : rows - 1;
  }
  rows = (rows / o.align_rows) * o.align_rows;
  if (rows < o.align_rows) rows = o.align_rows;
  o.rpt_max = rows;
  o.red_need = rows * M * o.cp;
}

struct Plan {
  int stage_target, stages, stage_w, stage_s, red_floats, kb;
  bool wide;   // 64 KB table, partial sums in its gaps
  PLayout L;
};

// Layout of a set of GEMVs at batch M (independent of the tiling, which never exceeds rpt_max):
// the fixed parts, then as many ring stages (2 ... kMaxStages) as shared memory holds; the stage
// size steps down from kStageTarget until two stages fit.  All GEMVs must share the k-block
// width (scale blocks of 32, or of 64 and more).
static bool plan_layout_with(int fmt, int M, const Job* jobs, int n, bool wide, Plan& P) {
  P.kb = kb_of(jobs[0].bs);
  P.wide = wide;
  for (int i = 0; i < n; ++i)
    if (kb_of(jobs[i].bs) != P.kb || !shape_ok(jobs[i].K, jobs[i].bs)) return false;
  for (P.stage_target = kStageTarget; P.stage_target >= 2048; P.stage_target = P.stage_target * 3 / 4) {
    P.stage_w = 1024; P.stage_s = 16; P.red_floats = 4;
    bool fits = true;
    for (int i = 0; i < n && fits; ++i) {
      GeomG gg;
      tile_rows(fmt, M, jobs[i].K, jobs[i].bs, P.stage_target, wide, gg);
      if (gg.red_need > kRedCapFloats) fits = false;
      if (wide && gg.rpt_max * gaps_per_output(gg.nspan) > kGapsPerBuf) fits = false;
      P.stage_w = max(P.stage_w, stage_bytes(gg.nbox, gg.rpt_max));
      P.stage_s = max(P.stage_s, ((gg.rpt_max * gg.srb) + 15) & ~15);
      P.red_floats = max(P.red_floats, gg.red_need);
    }
    if (!fits) continue;
    P.red_floats = (P.red_floats + kRedSlackFloats + 3) & ~3;
    for (P.stages = kMaxStages; P.stages >= 2; --P.stages) {
      P.L = playout(P.stages, P.stage_w, P.stage_s, P.red_floats, wide);
      if (P.L.total + 1024 <= kSmemCap) return true;   // + the 1 KB alignment slack
    }
  }
  return false;
}

// The 64 KB table at batch 1 when it leaves the same stage budget as the 32 KB table (its gaps
// take the partial sums), else the 32 KB table.
static bool plan_layout(int fmt, int M, const Job* jobs, int n, Plan& P) {
  if (M == 1) {
    Plan W, N;
    const bool w_ok = plan_layout_with(fmt, M, jobs, n, true, W);
    const bool n_ok = plan_layout_with(fmt, M, jobs, n, false, N);
    if (w_ok && (!n_ok || (W.stage_target >= N.stage_target && W.stages >= 2))) {
      P = W;
      return true;
    }
    if (n_ok) {
      P = N;
      return true;
    }
    return false;
  }
  return plan_layout_with(fmt, M, jobs, n, false, P);
}

int simt_max_batch(int format, int K, int bs) {
  Job jb{nullptr, nullptr, nullptr, nullptr, 1, K, bs, 0};
  for (int m : {8, 4, 2, 1}) {
    Plan P;
    if (plan_layout(format, m, &jb, 1, P)) return m;
  }
  return 0;
}

bool plan_simt(int format, int M, int K, int bs, SimtPlan* out) {
  const int mb = simt_max_batch(format, K, bs);
  if (mb < 1 || M < 1) return false;
  // the widest launch: min(M, mb) batch rows
  const int mm = M < mb ? M : mb;
  Job jb{nullptr, nullptr, nullptr, nullptr, 1, K, bs, 0};
  Plan P;
  if (!plan_layout(format, mm, &jb, 1, P)) return false;
  out->mb = mm;
  out->launches = (M + mb - 1) / mb;
  out->threads = kThreads;
  out->smem = P.L.total + 1024;
  out->stages = P.stages;
  return true;
}

// Everything a launch needs, computed on the host: parameters, the levels and GEMVs with their
// tiling, the tensor map of each GEMV (box rows = its rows per tile), and the geometry.
struct Prepared {
  PParams p;
  std::vector<PLevel> lv;
  std::vector<PGemv> gm;
  std::vector<CUtensorMap> maps;
  Plan plan;
  int grid;
};

static cudaError_t prepare(int fmt, const Job* jobs, int n, int M, const float* codebook, Prepared& P) {
  int nlev = 0;
  for (int i = 0; i < n; ++i) nlev = max(nlev, jobs[i].level + 1);
  if (n < 1 || n > kStepMaxGemvs || nlev > n) return cudaErrorNotSupported;
  if (!plan_layout(fmt, M, jobs, n, P.plan)) return cudaErrorNotSupported;
  const int gmax = device_sm_count();   // one CTA per SM: the ring is sized for the whole SM
  P.lv.assign((size_t)nlev, PLevel{});
  P.gm.assign((size_t)n, PGemv{});
  P.maps.assign((size_t)n, CUtensorMap{});
  PParams& p = P.p;
  p = PParams{};
  p.codebook = codebook;
  p.fmt = fmt;
  p.nlevels = nlev;
  p.ngemvs = n;
  p.M = M;
  p.stages = P.plan.stages; p.stage_w = P.plan.stage_w; p.stage_s = P.plan.stage_s;
  p.red_floats = P.plan.red_floats;
  // tiling, level by level: balanced tiles per CTA, rows per tile within each GEMV's stage budget
  int tile = 0, max_level_tiles = 0;
  for (int Lv = 0, i = 0; Lv < nlev; ++Lv) {
    const int first = i;
    long long rows = 0;
    int rmin = 1 << 30;
    while (i < n && jobs[i].level == Lv) {
      GeomG gg;
      tile_rows(fmt, M, jobs[i].K, jobs[i].bs, P.plan.stage_target, P.plan.wide, gg);
      rows += jobs[i].N;
      rmin = min(rmin, gg.rpt_max);
      ++i;
    }
    PLevel& lv = P.lv[(size_t)Lv];
    lv.gemv0 = first;
    lv.wait = Lv > 0 ? min(gmax, P.lv[(size_t)Lv - 1].ntiles) : 0;
    lv.tile0 = tile;
    const long long tpc = (rows + (long long)gmax * rmin - 1) / ((long long)gmax * rmin);
    for (int q = first; q < i; ++q) {
      GeomG gg;
      tile_rows(fmt, M, jobs[q].K, jobs[q].bs, P.plan.stage_target, P.plan.wide, gg);
      int rpt = (int)((rows + (long long)gmax * tpc - 1) / ((long long)gmax * tpc));
      if (rpt > 16) rpt = (rpt + 15) & ~15;                          // whole MMA row groups
      rpt = ((rpt + gg.align_rows - 1) / gg.align_rows) * gg.align_rows;
      rpt = min(rpt, gg.rpt_max);
      PGemv& g = P.gm[(size_t)q];
      g.packed = jobs[q].packed; g.scales = jobs[q].scales; g.x = jobs[q].x; g.y = jobs[q].y;
      g.tmap = nullptr;
      g.N = jobs[q].N; g.K = jobs[q].K; g.bs = jobs[q].bs; g.rpt = rpt;
      g.tile0 = tile; g.ntiles = (g.N + rpt - 1) / rpt; g.srb = gg.srb;
      g.nspan = gg.nspan; g.nbox = gg.nbox; g.slot = span_slot(rpt); g.cp = gg.cp;
      if (!encode_tmap_2d(&P.maps[(size_t)q], 1, g.packed, g.K / 2, g.N, kBoxK / 2, rpt)) return cudaErrorNotSupported;
      tile += g.ntiles;
    }
    lv.ntiles = tile - lv.tile0;
    max_level_tiles = max(max_level_tiles, lv.ntiles);
  }
  P.grid = nlev > 1 ? gmax : min(gmax, max_level_tiles);
  p.map1 = P.maps[0];
  p.lv1 = P.lv[0];
  p.gm1 = P.gm[0];
  return cudaSuccess;
}

template <int KB, bool SC32, int NSCF, bool WIDE>
static cudaError_t launch_prepared(Prepared& P, unsigned* counters, bool pdl, cudaStream_t stream) {
  auto kern = w4_persistent_kernel<KB, SC32, NSCF, WIDE>;
  static FuncAttrCache attrs;   // one per instance
  cudaError_t ea = attrs.ensure([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap); });
  if (ea != cudaSuccess) return ea;
  PParams& p = P.p;
  if (p.nlevels > 1 && !counters) return cudaErrorInvalidValue;
  if (p.ngemvs > 1 && (!p.lvt || !p.gmt)) return cudaErrorInvalidValue;
  p.counters = p.nlevels > 1 ? counters : nullptr;
  p.inject_timeout = take_fault_injection();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.grid);
  cfg.blockDim = dim3((unsigned)kThreads);
  cfg.dynamicSmemBytes = (size_t)P.plan.L.total + 1024;
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

// The instance for the launch's format, k-block width, scales per span (0 when the GEMVs' block
// sizes differ) and table.
template <bool WIDE>
static cudaError_t dispatch_table(int fmt, Prepared& P, unsigned* counters, bool pdl, cudaStream_t s) {
  int bs = P.gm[0].bs;
  for (const PGemv& g : P.gm)
    if (g.bs != bs) bs = 0;
  const int nsc = bs == 0 ? 0 : (bs >= kSpanK ? 1 : kSpanK / bs);
  if (P.plan.kb == 32) {   // block size 32: four scales per span
    if (fmt == 0) return launch_prepared<32, true, 4, WIDE>(P, counters, pdl, s);
    return launch_prepared<32, false, 4, WIDE>(P, counters, pdl, s);
  }
  if (fmt == 0) {
    if (nsc == 2) return launch_prepared<64, true, 2, WIDE>(P, counters, pdl, s);
    if (nsc == 1) return launch_prepared<64, true, 1, WIDE>(P, counters, pdl, s);
    return launch_prepared<64, true, 0, WIDE>(P, counters, pdl, s);
  }
  if (nsc == 2) return launch_prepared<64, false, 2, WIDE>(P, counters, pdl, s);
  if (nsc == 1) return launch_prepared<64, false, 1, WIDE>(P, counters, pdl, s);
  return launch_prepared<64, false, 0, WIDE>(P, counters, pdl, s);
}

static cudaError_t dispatch(int fmt, Prepared& P, unsigned* counters, bool pdl, cudaStream_t s) {
  if (P.plan.wide) return dispatch_table<true>(fmt, P, counters, pdl, s);
  return dispatch_table<false>(fmt, P, counters, pdl, s);
}

cudaError_t launch_gemv_simt(int format, const uint8_t* packed, const void* scales, const float* codebook,
                             const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                             cudaStream_t stream) {
  if (M < 1 || M > 8) return cudaErrorNotSupported;
  Job jb{packed, scales, x, y, N, K, bs, 0};
  Prepared P;
  cudaError_t e = prepare(format, &jb, 1, M, codebook, P);
  if (e != cudaSuccess) return e;
  return dispatch(format, P, nullptr, pdl, stream);
}

// Device tables of a multi-GEMV launch, at a 128-byte aligned base: the n tensor maps (128 bytes
// each), the levels (16 bytes each, at most n of them, padded to 128 bytes), the GEMVs.
static size_t tables_levels_off(int n) { return (size_t)n * sizeof(CUtensorMap); }
static size_t tables_gemvs_off(int n) { return tables_levels_off(n) + (((size_t)n * sizeof(PLevel) + 127) & ~(size_t)127); }
size_t step_tables_bytes(int n) { return tables_gemvs_off(n) + (size_t)n * sizeof(PGemv); }

static cudaError_t prepare_step(int format, const StepJob* jobs, int n, int M, const float* codebook, Prepared& P) {
  if (M < 1 || M > 8 || n < 1 || n > kStepMaxGemvs) return cudaErrorNotSupported;
  std::vector<Job> js((size_t)n);
  for (int i = 0; i < n; ++i) {
    js[(size_t)i] = Job{jobs[i].packed, jobs[i].scales, jobs[i].x, jobs[i].y, jobs[i].N, jobs[i].K, jobs[i].bs,
                        jobs[i].level};
  }
  return prepare(format, js.data(), n, M, codebook, P);
}

cudaError_t step_simt_tables(int format, const StepJob* jobs, int n, int M, const void* dev_base, void* blob) {
  Prepared P;
  cudaError_t e = prepare_step(format, jobs, n, M, nullptr, P);
  if (e != cudaSuccess) return e;
  uint8_t* out = static_cast<uint8_t*>(blob);
  memset(out, 0, step_tables_bytes(n));
  const uintptr_t base = reinterpret_cast<uintptr_t>(dev_base);
  for (int q = 0; q < n; ++q) P.gm[(size_t)q].tmap = reinterpret_cast<const CUtensorMap*>(base + (size_t)q * sizeof(CUtensorMap));
  memcpy(out, P.maps.data(), (size_t)n * sizeof(CUtensorMap));
  memcpy(out + tables_levels_off(n), P.lv.data(), P.lv.size() * sizeof(PLevel));
  memcpy(out + tables_gemvs_off(n), P.gm.data(), (size_t)n * sizeof(PGemv));
  return cudaSuccess;
}

cudaError_t launch_step_simt(int format, const StepJob* jobs, int n, int M, const float* codebook, unsigned* counters,
                             const void* dev_tables, bool pdl, cudaStream_t stream) {
  Prepared P;
  cudaError_t e = prepare_step(format, jobs, n, M, codebook, P);
  if (e != cudaSuccess) return e;
  const uint8_t* base = static_cast<const uint8_t*>(dev_tables);
  P.p.lvt = reinterpret_cast<const PLevel*>(base + tables_levels_off(n));
  P.p.gmt = reinterpret_cast<const PGemv*>(base + tables_gemvs_off(n));
  return dispatch(format, P, counters, pdl, stream);
}

// ---------------------------------------------------------------------------------------------
// Counters and tables for w4_gemv_levels_noalloc: fixed arrays inside the library, for callers that
// cannot allocate device memory.  In host code the names are only stand-ins for the device
// objects; their device addresses are looked up once per device and cached.
constexpr int kNoAllocMaxLevels = 256;
constexpr size_t kNoAllocTableBytes = (size_t)kStepMaxGemvs * (sizeof(CUtensorMap) + sizeof(PLevel) + sizeof(PGemv));
static __device__ __align__(256) unsigned int g_noalloc_counters[kNoAllocMaxLevels + 1];
static __device__ __align__(128) uint4 g_noalloc_tables[kNoAllocTableBytes / 16];

static cudaError_t noalloc_arrays(unsigned** counters, void** tables) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  // the addresses belong to the context they were looked up in: look them up again when the
  // device's context has changed (cudaDeviceReset)
  const unsigned long long ctx = current_context_id();
  static std::mutex mu;
  static unsigned* caddr[kMaxDevices] = {};
  static void* taddr[kMaxDevices] = {};
  static unsigned long long cid[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (caddr[dev] == nullptr || ctx == 0 || cid[dev] != ctx) {
    void* pc = nullptr;
    void* pt = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&pc, g_noalloc_counters);   // with this device current
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(&pt, g_noalloc_tables);
    if (e != cudaSuccess) return e;
    caddr[dev] = static_cast<unsigned*>(pc);
    taddr[dev] = pt;
    cid[dev] = ctx;
  }
  *counters = caddr[dev];
  *tables = taddr[dev];
  return cudaSuccess;
}

int noalloc_max_levels() { return kNoAllocMaxLevels; }

cudaError_t launch_step_simt_noalloc(int format, const StepJob* jobs, int n, int M, const float* codebook,
                                     int nlevels, cudaStream_t stream) {
  if (nlevels < 1 || nlevels > kNoAllocMaxLevels || n > kStepMaxGemvs) return cudaErrorInvalidValue;
  static_assert(kNoAllocTableBytes >= kStepMaxGemvs * sizeof(CUtensorMap) + kStepMaxGemvs * sizeof(PLevel) +
                                          kStepMaxGemvs * sizeof(PGemv), "no-alloc table array too small");
  unsigned* counters = nullptr;
  void* tables = nullptr;
  cudaError_t e = noalloc_arrays(&counters, &tables);
  if (e != cudaSuccess) return e;
  // the arrays keep the previous call's contents: this call's tables, and counters from zero
  std::vector<uint8_t> blob(step_tables_bytes(n));
  e = step_simt_tables(format, jobs, n, M, tables, blob.data());
  if (e == cudaSuccess) e = cudaMemcpyAsync(tables, blob.data(), blob.size(), cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(counters, 0, sizeof(unsigned) * (size_t)(nlevels + 1), stream);
  if (e == cudaSuccess) e = launch_step_simt(format, jobs, n, M, codebook, counters, tables, true, stream);
  return e;
}

unsigned int read_clear_error_persist() { return read_clear_error_word_here(); }

}  // namespace w4
