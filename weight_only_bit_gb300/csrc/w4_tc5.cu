// w4_tc5.cu -- fused 4-bit dequant-GEMM on the 5th-generation tensor cores (tcgen05) for batches
// 9 ... 256 (sm_103a).
//
// At these batches every decoded weight feeds 9-128 multiply-adds: the work is a dense
// contraction and belongs on the tensor cores ("My Triton Kernel Ties bitsandbytes", section "Why
// Marlin is still faster").  Weights are decoded on chip and never written back to DRAM ("LLM
// Quantization on RTX 4060", section "Fused Kernel: Moving Dequantization On-Chip").
//
// y^T[N][M] = W_hat[N][K] . x^T[K][M], one CTA per SM taking tiles of 128 weight rows in turn:
//   * packed weights: one TMA tensor copy per 256-k super-chunk brings 128 rows x 128 bytes (16 KB)
//     into a ring of shared-memory slots, 128-byte swizzled so that the decoders' reads are free
//     of bank conflicts;
//   * A = 128 weight rows x 64 k per stage, decoded by 512 threads (byte-pair table of
//     w4_decode.cuh: NF4 code values, q - 8 for INT4, E2M1 values for FP4; times the block scale
//     in FP16) and
//     stored straight into tensor memory (tcgen05.st): lane = weight row, 32 columns per stage,
//     two FP16 k values per column.  The MMA reads A from tensor memory, so decoded weights never
//     pass through shared memory (whose bandwidth the byte-pair table already uses);
//   * B = x: one TMA tensor copy per 64-k stage, NB rows (rows M ... NB - 1 filled with zero by
//     the copy), 128-byte swizzled, which is the canonical K-major SW128 operand layout;
//   * D = FP32 accumulators in tensor memory: 128 lanes (weight rows) x NB columns, two of them so
//     that the epilogue of one tile overlaps the MMAs of the next (NB <= 128), or one of 256
//     columns for prefill-sized batches (NB = 256: each weight tile is decoded and read once per
//     256 batch rows; the MMA's N is 256);
//   * one thread issues four tcgen05.mma.cta_group::1.kind::f16 per stage (K = 16 each) and
//     commits them to the stage's "empty" barrier; after a tile's last stage, to the
//     accumulator's "full" barrier;
//   * epilogue: tcgen05.ld of each warp's 32 lanes, rounded to FP16, written to y.
// Split-K (when the row tiles alone cannot fill the SMs): the super-chunks of a tile are divided
// among the ks CTAs of a thread-block cluster; each CTA leaves its FP32 partial tile in its (by
// then idle) x stages, and after a cluster barrier CTA r sums its share of the rows over the
// cluster in rank order through distributed shared memory: no global scratch, and the result does
// not depend on timing.
// Block scales: per super-chunk, one scale warp per packed slot loads the slot's 128 x (256 / bs)
// scales, rounds them to FP16 pairs and stores them next to the slot, so the decoders touch no
// global memory (the producer asks L2 to prefetch each tile's scale block, one contiguous range).
// Every mbarrier wait is bounded; a lost wait is recorded in the device error word, and the
// kernel still waits (bounded) for its own copies and MMAs and frees its tensor memory.
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <mutex>

#include "w4_common.cuh"
#include "w4_decode.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr int kT5Rows = 128;                 // weight rows per tile (the MMA's M)
constexpr int kT5Kc = 64;                    // k per stage
constexpr int kT5Sk = 256;                   // k per packed super-chunk (128 bytes per row)
constexpr int kT5CPS = kT5Sk / kT5Kc;        // stages per super-chunk
constexpr uint32_t kT5AccCols = 256;         // tensor memory: columns 0 ... 255 accumulators,
constexpr uint32_t kT5ACols = kT5Kc / 2;      // then A stages of 32 columns each
constexpr int kT5MaxStages = (512 - kT5AccCols) / kT5ACols;   // 8
constexpr int kT5PBytes = kT5Rows * kT5Sk / 2;   // 16 KB
constexpr int kT5SStride = kT5Rows * 4 + 32;   // bytes per scale index j in a scale slot (padded)
constexpr int kT5SBytes = 8 * kT5SStride;        // up to 8 scales per row per super-chunk (bs = 32)
constexpr uint32_t kT5Sbo = 1024;            // B: 8-row groups of 128 bytes

struct T5Params {
  CUtensorMap tm_packed;   // uint8 [N][K/2], box 128 x 128, 128-byte swizzle
  CUtensorMap tm_x;        // fp16 [M][K], box 64 x NB, 128-byte swizzle
  const __half* tm_x_base; // x (the map over it is made per batch tile width)
  const void* scales;
  const float* codebook;
  __half* y;
  int M, N, K, bs;
  int ks;            // CTAs per cluster along K (1: persistent over row tiles)
  int nchunk;        // K / kT5Kc
  int nsc;           // super-chunks per tile
  int stages;        // x / A stages
  int np;            // packed slots
  int inject_timeout;  // test hook: the packed producer issues no copies (every wait then runs out)
};

// Shared-memory matrix descriptor of B (version 1): 128-byte swizzle (layout type 2 in bits 61-63),
// SBO = 8 rows of 128 bytes, LBO unused; a K = 16 step moves the start address by 32 bytes inside
// the swizzle atom.
__device__ __forceinline__ uint64_t t5_desc_b(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)((kT5Sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: FP32 D, FP16 A and B, both K-major, M = 128, N = NB.
template <int NB>
__host__ __device__ constexpr uint32_t t5_idesc() {
  return (1u << 4) | ((uint32_t)(NB >> 3) << 17) | ((uint32_t)(kT5Rows >> 4) << 24);
}

// D[tmem] (+)= A[tmem] . B[smem]^T, M = 128, K = 16.
__device__ __forceinline__ void t5_mma_ts(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      ::"r"(dtmem), "r"(atmem), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

// This warp's 32 lanes x 8 consecutive columns of tensor memory <- 8 registers per thread.
__device__ __forceinline__ void t5_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void t5_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void t5_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void t5_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive FP32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void t5_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2-D TMA tensor copy global -> shared; completion adds the box's bytes to `bar`.
__device__ __forceinline__ void t5_tma2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void t5_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t t5_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void t5_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Four floats (16-byte aligned) from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float4 t5_ld_dsmem4(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote)
               : "memory");
  return v;
}

// Partial tiles of a split: [row][NB + 4] floats (rows 16-byte aligned).
__host__ __device__ constexpr int t5_part_stride_rt(int NB) { return NB + 4; }
template <int NB>
__host__ __device__ constexpr int t5_part_stride() { return t5_part_stride_rt(NB); }

__device__ __forceinline__ uint64_t t5_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Warp roles (one CTA per SM):
//   warp 0   packed producer (one lane): a TMA copy per super-chunk into NP slots, L2 evict-first;
//            asks L2 to prefetch each tile's scale block one tile ahead;
//   warp 1   x producer (one lane): a TMA copy of x per stage into NS stages, L2 evict-last;
//   warp 2   tensor-memory owner and MMA issuer (one lane);
//   warps 3 ... 6    scale warps: warp 3 + i fills the scales of packed slot i;
//   warps 7 ... 22   decoders: warp w owns tensor-memory lanes (= tile rows) 32 (w % 4) ... + 31
//                    and k quarter (w - 7) / 4 of each stage: each thread turns the 16 weights of
//                    its row and quarter into FP16 and stores them to its lane, two stages per step;
//   warps 23 ... 26  epilogue: tensor memory -> FP16 y; then the accumulator is released.
constexpr int kT5Pw = 0, kT5Xw = 1, kT5Mw = 2, kT5S0 = 3, kT5Sw = 4, kT5Dq0 = 7, kT5Dq = 16, kT5Ep0 = 23, kT5Ep = 4;
constexpr int kT5Threads = (kT5Ep0 + kT5Ep) * 32;     // 864

struct T5Layout {
  int np, ns, packed, sc, xb, xstage, bar, total;
};

// Offsets from a 1024-byte aligned base (the swizzled TMA destinations need that alignment).
__host__ __device__ inline T5Layout t5_layout(int NB, int NP, int NS) {
  T5Layout L;
  L.np = NP;
  L.ns = NS;
  L.packed = kLutBytes;                                // 32 KB table, then NP x 16 KB slots
  L.xstage = NB * kT5Kc * 2;                          // x: NB rows x 128 bytes
  L.sc = L.packed + NP * kT5PBytes;                  // NP scale slots
  L.xb = L.sc + ((NP * kT5SBytes + 1023) & ~1023);
  L.bar = L.xb + NS * L.xstage;
  L.total = L.bar + (2 * NP + 3 * NS + 5) * 8 + 16;
  return L;
}

template <int NB>
__host__ __device__ constexpr int t5_tmem_cols() { return NB < 32 ? 32 : NB; }
// Accumulators in tensor memory: two (the epilogue of one tile overlaps the MMAs of the next) up
// to 128 batch columns; one of 256 columns (the whole accumulator half of tensor memory) at 256.
template <int NB>
__host__ __device__ constexpr int t5_nacc() { return NB <= 128 ? 2 : 1; }

// Bounded wait on an mbarrier phase for the pipeline roles.
__device__ __forceinline__ bool t5_wait(uint64_t* bar, uint32_t parity, uint32_t site) {
  return mbar_wait(bar, parity, site);
}

// A ring position: index and phase parity, advanced without divisions.
struct T5Ring {
  int i, ph;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) { i = 0; ph ^= 1; }
  }
};

// Block scale of (row, k) as FP16 (NF4: the FP32 absmax rounded to nearest).
template <int FMT>
__device__ __forceinline__ uint32_t t5_scale_bits(const void* scales, long long idx) {
  if (FMT == 0) {
    return __half_as_ushort(__float2half_rn(__ldg(reinterpret_cast<const float*>(scales) + idx)));
  }
  return __ldg(reinterpret_cast<const unsigned short*>(scales) + idx);
}

template <int FMT, int NB>
__global__ void __launch_bounds__(kT5Threads, 1) w4_tc5_kernel(const __grid_constant__ T5Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const T5Layout Lo = t5_layout(NB, p.np, p.stages);
  const int NP = Lo.np, NS = Lo.ns;
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem);
  uint64_t* pfull = reinterpret_cast<uint64_t*>(smem + Lo.bar);   // packed slot landed
  uint64_t* pempty = pfull + NP;                                  // packed slot read by all decoders
  uint64_t* xfull = pempty + NP;                                  // stage's x landed
  uint64_t* afull = xfull + NS;                                   // stage's A decoded
  uint64_t* sempty = afull + NS;                                  // stage's MMAs complete
  uint64_t* accfull = sempty + NS;                                // accumulator b complete
  uint64_t* accempty = accfull + 2;                               // accumulator b read out
  uint64_t* mmadone = accempty + 2;                               // every MMA of this CTA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mmadone + 1);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nrb = (p.N + kT5Rows - 1) / kT5Rows;
  const int nck = p.nchunk;
  // tiles taken in turn by the CTAs (ks == 1), or one tile per cluster with the super-chunks
  // [s0, s1) of it for this CTA (ks > 1)
  const int ks = p.ks;
  const uint32_t rank = ks > 1 ? t5_cluster_rank() : 0u;
  const int tile0 = ks > 1 ? (int)blockIdx.x / ks : (int)blockIdx.x;
  const int tstep = ks > 1 ? nrb : (int)gridDim.x;
  const int s0 = ks > 1 ? (int)rank * p.nsc / ks : 0;
  const int s1 = ks > 1 ? ((int)rank + 1) * p.nsc / ks : p.nsc;
  const int c0 = s0 * kT5CPS, c1 = min(s1 * kT5CPS, nck);
  const int spr = p.K / p.bs;
  constexpr int kCols = t5_tmem_cols<NB>();
  constexpr int kEs = FMT == 0 ? 4 : 2;   // bytes per scale

  // ---- set-up: table, barriers, tensor memory
  build_lut(lut, FMT, p.codebook, tid, kT5Threads);
  if (tid == 0) {
    for (int i = 0; i < NP; ++i) {
      mbar_init(&pfull[i], 2);          // the TMA producer (with the bytes) and the scale warp
      mbar_init(&pempty[i], kT5Dq);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&xfull[i], 1);
      mbar_init(&afull[i], kT5Dq);
      mbar_init(&sempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], kT5Ep);
    }
    mbar_init(mmadone, 1);
    fence_mbar_init();
  }
  if (warp == kT5Mw) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tmem_slot)), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  t5_fence_before();
  __syncthreads();
  t5_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  bool ok = true;

  if (warp == kT5Pw) {
    // ================================================================ packed producer
    if (lane == 0 && !p.inject_timeout) {
      const uint64_t pol = policy_evict_first();
      const uint32_t pk = smem_u32(smem + Lo.packed);
      auto prefetch_scales = [&](int rb) {
        if (rb >= nrb) return;
        const int rows = min(kT5Rows, p.N - rb * kT5Rows);
        const uint32_t bytes = (uint32_t)((long long)rows * spr * kEs) & ~15u;
        if (bytes > 0)
          t5_prefetch_l2(reinterpret_cast<const uint8_t*>(p.scales) + (size_t)rb * kT5Rows * spr * kEs, bytes);
      };
      prefetch_scales(tile0);
      T5Ring ps{0, 0};
      int jp = 0;
      for (int rb = tile0; rb < nrb && ok; rb += tstep) {
        prefetch_scales(rb + tstep);
        for (int s = s0; s < s1 && ok; ++s, ++jp) {
          if (jp >= NP) ok = t5_wait(&pempty[ps.i], ps.ph ^ 1, 0x311);
          if (!ok) break;
          mbar_arrive_expect_tx(&pfull[ps.i], kT5PBytes);
          t5_tma2d(pk + ps.i * kT5PBytes, &p.tm_packed, s * (kT5Sk / 2), rb * kT5Rows, &pfull[ps.i], pol);
          ps.next(NP);
        }
      }
      // every copy issued has landed before the CTA may exit (normally long since consumed)
      T5Ring q = ps;
      for (int n = 0; n < min(jp, NP); ++n) {
        q.i = q.i == 0 ? NP - 1 : q.i - 1;
        if (q.i == NP - 1) q.ph ^= 1;
        t5_wait(&pfull[q.i], q.ph, 0x319);
      }
    }
    __syncwarp();
  } else if (warp == kT5Xw) {
    // ================================================================ x producer
    if (lane == 0) {
      const uint64_t pol = t5_policy_evict_last();
      T5Ring ss{0, 0};
      int jj = 0;
      for (int rb = tile0; rb < nrb && ok; rb += tstep) {
        for (int c = c0; c < c1 && ok; ++c, ++jj) {
          if (jj >= NS) ok = t5_wait(&sempty[ss.i], ss.ph ^ 1, 0x312);
          if (!ok) break;
          mbar_arrive_expect_tx(&xfull[ss.i], NB * kT5Kc * 2);
          t5_tma2d(smem_u32(smem + Lo.xb + ss.i * Lo.xstage), &p.tm_x, c * kT5Kc, 0, &xfull[ss.i], pol);
          ss.next(NS);
        }
      }
      T5Ring q = ss;
      for (int n = 0; n < min(jj, NS); ++n) {
        q.i = q.i == 0 ? NS - 1 : q.i - 1;
        if (q.i == NS - 1) q.ph ^= 1;
        t5_wait(&xfull[q.i], q.ph, 0x31a);
      }
    }
    __syncwarp();
  } else if (warp == kT5Mw) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = t5_idesc<NB>();
      T5Ring ss{0, 0};
      int tile = 0;
      constexpr int NACC = t5_nacc<NB>();
      for (int rb = tile0; rb < nrb && ok; rb += tstep, ++tile) {
        const int b = tile % NACC;
        if (tile >= NACC) ok = t5_wait(&accempty[b], ((tile / NACC) - 1) & 1, 0x313);
        t5_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * kCols);
        for (int c = c0; c < c1 && ok; ++c) {
          ok = t5_wait(&afull[ss.i], ss.ph, 0x314) && t5_wait(&xfull[ss.i], ss.ph, 0x315);
          if (!ok) break;
          t5_fence_after();
          const uint32_t ta = tmem + kT5AccCols + (uint32_t)ss.i * kT5ACols;
          const uint32_t sb = smem_u32(smem + Lo.xb + ss.i * Lo.xstage);
#pragma unroll
          for (int q = 0; q < kT5Kc / 16; ++q) {
            t5_mma_ts(d, ta + q * 8, t5_desc_b(sb + q * 32), idesc, (c > c0 || q > 0) ? 1u : 0u);
          }
          t5_commit(&sempty[ss.i]);
          ss.next(NS);
        }
        if (ok) t5_commit(&accfull[b]);
      }
      // every MMA issued is complete before tensor memory is freed
      t5_commit(mmadone);
      t5_wait(mmadone, 0, 0x31b);
    }
    __syncwarp();
  } else if (warp < kT5Dq0) {
    // ================================================================ scale warps
    const int w = warp - kT5S0;
    if (w < NP) {
      const int S = kT5Sk / p.bs;                      // scales per row per super-chunk (1 ... 8)
      const int lgS = 31 - __clz(S);
      const uint32_t sslot = smem_u32(smem + Lo.sc + w * kT5SBytes);
      int jp = 0;
      for (int rb = tile0; rb < nrb && ok; rb += tstep) {
        const int valid = min(kT5Rows, p.N - rb * kT5Rows);
        for (int s = s0; s < s1 && ok; ++s, ++jp) {
          if (jp % NP != w) continue;
          const int use = jp / NP;
          if (use >= 1) ok = t5_wait(&pempty[w], (use - 1) & 1, 0x31c);
          if (!ok) break;
          // value v = row * S + j: scale j of the super-chunk for row `row`; 16 loads in flight
          // per lane, in one or two rounds
          for (int base = 0; base < 4 * S; base += 16) {
            uint32_t h[16];
#pragma unroll
            for (int it = 0; it < 16; ++it) {
              h[it] = 0u;
              const int v = (base + it) * 32 + lane;
              const int row = v >> lgS, j = v & (S - 1);
              if (base + it < 4 * S && row < valid && s * S + j < spr)
                h[it] = t5_scale_bits<FMT>(p.scales, (long long)(rb * kT5Rows + row) * spr + s * S + j);
            }
#pragma unroll
            for (int it = 0; it < 16; ++it) {
              const int v = (base + it) * 32 + lane;
              if (base + it < 4 * S) {
                const int row = v >> lgS, j = v & (S - 1);
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(sslot + j * kT5SStride + row * 4), "r"(h[it] | (h[it] << 16))
                             : "memory");
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&pfull[w]);
        }
      }
    }
    __syncwarp();
  } else if (warp < kT5Ep0) {
    // ================================================================ decoders
    const int quarter = warp & 3;                        // tensor-memory lanes 32 quarter ... + 31
    const int h = (warp - kT5Dq0) >> 2;                  // k 16h ... 16h + 15 of each stage
    const int r = quarter * 32 + lane;                   // row within the tile
    const uint32_t lut_lane = smem_u32(lut) + (uint32_t)lane * 4u;
    const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16) + kT5AccCols + (uint32_t)h * 8u;
    const int lgbs = 31 - __clz(p.bs);
    T5Ring ps{0, 0}, ss{0, 0};
    int jj = 0;
    // 16 weights (8 packed bytes) with FP16 scale pair `sc` -> 8 FP16 pairs in tensor memory
    auto decode = [&](uint2 wv, uint32_t sc, uint32_t taddr) {
      const uint32_t w2[2] = {wv.x, wv.y};
      uint32_t hv[8];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t byte;
          asm("prmt.b32 %0, %1, 0, %2;" : "=r"(byte) : "r"(w2[g]), "r"(0x4440 + b));
          const uint32_t c2 = lds32(lut_lane + byte * 128u);
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hv[4 * g + b]) : "r"(c2), "r"(sc));
        }
      }
      t5_st8(taddr, hv);
    };
    for (int rb = tile0; rb < nrb && ok; rb += tstep) {
      for (int s = s0; s < s1 && ok; ++s) {
        ok = t5_wait(&pfull[ps.i], ps.ph, 0x316);
        if (!ok) break;
        const uint8_t* slot = smem + Lo.packed + ps.i * kT5PBytes;
        const uint32_t sslot = smem_u32(smem + Lo.sc + ps.i * kT5SBytes) + (uint32_t)r * 4u;
        const int ncs = min(kT5CPS, nck - s * kT5CPS);
        for (int ci = 0; ci < ncs && ok; ci += 2) {
          const bool two = ci + 1 < ncs;
          T5Ring s1 = ss;
          s1.next(NS);
          if (jj >= NS) ok = t5_wait(&sempty[ss.i], ss.ph ^ 1, 0x317);
          if (ok && two && jj + 1 >= NS) ok = t5_wait(&sempty[s1.i], s1.ph ^ 1, 0x317);
          if (!ok) break;
          t5_fence_after();
          // bytes 32 c + 8 h ... + 7 of the row: 16-byte unit 2 c + h/2, swizzled by row & 7
          const uint32_t o0 = (uint32_t)r * 128u + ((uint32_t)((2 * ci + (h >> 1)) ^ (r & 7)) << 4) + (h & 1) * 8u;
          const uint32_t o1 = (uint32_t)r * 128u + ((uint32_t)((2 * ci + 2 + (h >> 1)) ^ (r & 7)) << 4) + (h & 1) * 8u;
          const uint2 w0 = *reinterpret_cast<const uint2*>(slot + o0);
          const uint2 w1 = two ? *reinterpret_cast<const uint2*>(slot + o1) : make_uint2(0, 0);
          const uint32_t sc0 = lds32(sslot + (uint32_t)(((ci * kT5Kc + h * 16) >> lgbs) * kT5SStride));
          const uint32_t sc1 = two ? lds32(sslot + (uint32_t)((((ci + 1) * kT5Kc + h * 16) >> lgbs) * kT5SStride)) : 0u;
          decode(w0, sc0, tlane + (uint32_t)ss.i * kT5ACols);
          if (two) decode(w1, sc1, tlane + (uint32_t)s1.i * kT5ACols);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");   // this warp's A columns written
          t5_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&afull[ss.i]);
            if (two) mbar_arrive(&afull[s1.i]);
          }
          ss = s1;
          ++jj;
          if (two) {
            ss.next(NS);
            ++jj;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[ps.i]);
        ps.next(NP);
      }
    }
  } else {
    // ================================================================ epilogue
    const int g = warp & 3;                          // tensor memory lanes 32g ... 32g + 31
    int tile = 0;
    constexpr int NACC = t5_nacc<NB>();
    for (int rb = tile0; rb < nrb && ok; rb += tstep, ++tile) {
      const int b = tile % NACC;
      ok = t5_wait(&accfull[b], (tile / NACC) & 1, 0x318);
      if (!ok) break;
      t5_fence_after();
      const uint32_t taddr = tmem + (uint32_t)(b * kCols) + ((uint32_t)(g * 32) << 16);
      const int orow = rb * kT5Rows + g * 32 + lane;
      // split: the partial row goes to this CTA's x stages (all consumed)
      float* part = reinterpret_cast<float*>(smem + Lo.xb) + (g * 32 + lane) * t5_part_stride<NB>();
#pragma unroll
      for (int n0 = 0; n0 < NB; n0 += 16) {
        float v[16];
        t5_ld16(taddr + (uint32_t)n0, v);
        if (ks > 1) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(part + n0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else if (orow < p.N) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (n0 + i < p.M) p.y[(size_t)(n0 + i) * p.N + orow] = __float2half_rn(v[i]);
          }
        }
      }
      t5_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[b]);
    }
  }
  // ---- teardown: every copy landed and every MMA complete (the producers and the MMA issuer
  // waited for their own work above)
  t5_fence_before();
  __syncthreads();
  if (ks > 1) {
    // CTA `rank` sums rows [r0, r1) of the tile over the cluster, in rank order
    t5_cluster_sync();
    const int rows_per = (kT5Rows + ks - 1) / ks;
    const int r0 = (int)rank * rows_per, r1 = min(kT5Rows, r0 + rows_per);
    const int nr = r1 - r0;
    const uint32_t pbase = smem_u32(smem + Lo.xb);
    const int m4 = (p.M + 3) >> 2;                     // groups of four batch rows
    for (int e = tid; e < nr * m4; e += kT5Threads) {
      const int n = (e / nr) * 4, row = r0 + e % nr;
      const int orow = tile0 * kT5Rows + row;
      if (orow < p.N) {
        const uint32_t a = pbase + (uint32_t)((row * t5_part_stride<NB>() + n) * 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < ks; ++c) {
          const float4 v = t5_ld_dsmem4(a, (uint32_t)c);
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        const float r4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n + i < p.M) p.y[(size_t)(n + i) * p.N + orow] = __float2half_rn(r4[i]);
      }
    }
    t5_cluster_sync();                   // the peers' reads of this CTA's partial are done
  }
  if (warp == kT5Mw) {
    t5_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// ---------------------------------------------------------------- host side

// Launch geometry of one GEMV on this kernel; host only, no device call.  False for shapes the
// kernel does not take.
bool plan_tc5(int M, int N, int K, int bs, int sms, Tc5Plan* o) {
  // block sizes 32 ... 256 (each thread's 16-k slice lies in one block); K whole 64-k stages
  if (M < 1 || M > 2 * kT5Rows || N < 1 || K < kT5Kc || K % kT5Kc != 0 || bs < 32 || sms < 1) return false;
  const int NB = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  // rings: 4 packed slots (64 KB of weights in flight per SM; 3 at 256 batch columns, whose x
  // stages are 32 KB) and up to 8 stages (the A stages fill the rest of tensor memory), as many as
  // fit in 227 KB with the 1 KB alignment slack
  const int NP = NB == 256 ? 3 : 4;
  static_assert(4 <= kT5Sw, "one scale warp per packed slot");
  int NS = 0;
  for (int ns = kT5MaxStages; ns >= 4 && NS == 0; --ns) {
    if (t5_layout(NB, NP, ns).total + 1024 <= 227 * 1024) NS = ns;
  }
  if (NS == 0) return false;
  const T5Layout L = t5_layout(NB, NP, NS);
  const int nrb = (N + kT5Rows - 1) / kT5Rows;
  const int nchunk = K / kT5Kc;
  const int nsc = (K + kT5Sk - 1) / kT5Sk;
  // split K over a cluster when the row tiles fill fewer than half the SMs: enough CTAs to cover
  // the SMs, at most 8 (a portable cluster) and at least one super-chunk each, and only when the
  // stages saved outweigh the split's cost.  Measured on GB300: a 64-k stage costs about 0.37 us;
  // a split costs about 3 us (cluster launch and barriers) plus 0.05 us per batch row (each CTA
  // reads 32 M float4s through distributed shared memory, whatever ks).  The partial tile must
  // fit in the x stages.
  int ks = 1;
  if (2 * nrb <= sms) {
    ks = min(8, min(sms / nrb, nsc));
    const double saved_us = 0.37 * nchunk * (1.0 - 1.0 / (ks > 0 ? ks : 1));
    if (ks < 2 || saved_us < 0.05 * M + 3.0 || NS * L.xstage < kT5Rows * t5_part_stride_rt(NB) * 4) ks = 1;
  }
  o->nb = NB;
  o->np = NP;
  o->ns = NS;
  o->ks = ks;
  o->grid = ks > 1 ? nrb * ks : min(nrb, sms);
  o->threads = kT5Threads;
  o->smem = L.total + 1024;
  return true;
}

template <int FMT, int NB>
static cudaError_t launch_tc5_nb(T5Params& p, const Tc5Plan& pl, bool pdl, cudaStream_t stream) {
  auto kern = w4_tc5_kernel<FMT, NB>;
  static FuncAttrCache attrs;
  cudaError_t ea = attrs.ensure([&] { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024); });
  if (ea != cudaSuccess) return ea;
  if (!encode_tmap_2d(&p.tm_x, 2, p.tm_x_base, p.K, p.M, kT5Kc, NB))
    return cudaErrorNotSupported;
  p.np = pl.np;
  p.stages = pl.ns;
  p.ks = pl.ks;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid);
  cfg.blockDim = dim3((unsigned)pl.threads);
  cfg.dynamicSmemBytes = (size_t)pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)pl.ks;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pl.ks > 1 ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  return e;
}

cudaError_t launch_gemv_tc5(int format, const uint8_t* packed, const void* scales, const float* codebook,
                            const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                            cudaStream_t stream) {
  Tc5Plan pl;
  // the TMA copies need 16-byte aligned bases
  if (!plan_tc5(M, N, K, bs, device_sm_count(), &pl) || (reinterpret_cast<uintptr_t>(packed) & 15) ||
      (reinterpret_cast<uintptr_t>(x) & 15))
    return cudaErrorNotSupported;
  T5Params p;
  if (!encode_tmap_2d(&p.tm_packed, 1, packed, K / 2, N, kT5Sk / 2, kT5Rows))
    return cudaErrorNotSupported;
  p.tm_x_base = x;
  p.scales = scales; p.codebook = codebook; p.y = y;
  p.M = M; p.N = N; p.K = K; p.bs = bs;
  p.nchunk = K / kT5Kc;
  p.nsc = (K + kT5Sk - 1) / kT5Sk;
  p.ks = 1;
  p.inject_timeout = take_fault_injection();
  switch (format * 1000 + pl.nb) {
    case 16: return launch_tc5_nb<0, 16>(p, pl, pdl, stream);
    case 32: return launch_tc5_nb<0, 32>(p, pl, pdl, stream);
    case 64: return launch_tc5_nb<0, 64>(p, pl, pdl, stream);
    case 128: return launch_tc5_nb<0, 128>(p, pl, pdl, stream);
    case 1016: return launch_tc5_nb<1, 16>(p, pl, pdl, stream);
    case 1032: return launch_tc5_nb<1, 32>(p, pl, pdl, stream);
    case 1064: return launch_tc5_nb<1, 64>(p, pl, pdl, stream);
    case 1128: return launch_tc5_nb<1, 128>(p, pl, pdl, stream);
    case 2016: return launch_tc5_nb<2, 16>(p, pl, pdl, stream);
    case 2032: return launch_tc5_nb<2, 32>(p, pl, pdl, stream);
    case 2064: return launch_tc5_nb<2, 64>(p, pl, pdl, stream);
    case 2128: return launch_tc5_nb<2, 128>(p, pl, pdl, stream);
    case 256: return launch_tc5_nb<0, 256>(p, pl, pdl, stream);
    case 1256: return launch_tc5_nb<1, 256>(p, pl, pdl, stream);
    case 2256: return launch_tc5_nb<2, 256>(p, pl, pdl, stream);
    default: return cudaErrorNotSupported;
  }
}

unsigned int read_clear_error_tc5() { return read_clear_error_word_here(); }

}  // namespace w4
