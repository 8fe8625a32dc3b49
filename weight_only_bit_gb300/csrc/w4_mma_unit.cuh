// w4_mma_unit.cuh -- the decode-and-multiply unit of the batch 1 ... 8 kernel: 16 weight rows x 128 k
// of a tile in shared memory, decoded through the byte-pair table into mma.sync.m16n8k16 A fragments
// (FP16 x FP16 -> FP32) against x, with the block scales applied to FP32 accumulators.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "w4_common.cuh"
#include "w4_decode.cuh"

namespace w4 {

constexpr int kSpanK = 128;            // k per unit of work (one partial sum per row and span)
constexpr int kBoxK = 256;             // k per TMA box (128 bytes of a row): two spans

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory loads by 32-bit shared address.  The table loads are plain asm: the table is
// constant once built, and each address depends on packed data loaded after the stage's wait.  The
// ring loads are volatile, so they stay after the wait that makes their data valid.
__device__ __forceinline__ uint32_t lds_table(uint32_t a) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_ring32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds_ring64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
// Shared-memory store that only lanes with `pred` perform (a predicated store, no branch).
__device__ __forceinline__ void sts_f32_if(uint32_t a, float v, bool pred) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p st.shared.f32 [%0], %1;\n}"
               ::"r"(a), "f"(v), "r"((int)pred) : "memory");
}
__device__ __forceinline__ float lds_scale32(uint32_t a) { return __uint_as_float(lds_ring32(a)); }
__device__ __forceinline__ float lds_scale16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return __half2float(__ushort_as_half(v));
}

// Decoded pair (element 2j in the low half) of packed byte b (0 ... 3) of word w, from this lane's
// copy of the byte-pair table.  32 KB table: lut = shared address of the lane's entry 0.  64 KB
// table (WIDE): lut = the table's shared address (the same in every lane) and lane4 = 4 * lane; one
// byte permute forms the entry's offset 256 * byte + lane4.
template <bool WIDE>
__device__ __forceinline__ uint32_t lut_pair(uint32_t lut, uint32_t lane4, uint32_t w, int b) {
  if (WIDE) {
    uint32_t off;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(off) : "r"(w), "r"(lane4), "r"(0x5504 | (b << 4)));
    return lds_table(lut + off);
  }
  uint32_t byte;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(byte) : "r"(w), "r"(0x4440 + b));
  return lds_table(lut + (byte << 7));
}

// Where a tile's span partials live.  Dense: output o's partial of span c at float o * cp + c of
// the buffer.  Gaps (the 64 KB table's 128-byte gaps, 32 floats each): output o owns hpo
// consecutive gaps from gap o * hpo, span c in gap c / 32 at word (c + 4 (o & 7)) mod 32 (the
// rotation puts eight consecutive outputs' runs of four spans in distinct banks); base = the
// buffer's first gap, gaps 256 bytes apart.  at(o, c) with c a multiple of 4 starts four
// consecutive spans (16-byte aligned).
struct PartDense {
  const float* base;
  int cp;
  __device__ __forceinline__ const float* at(int o, int c) const { return base + o * cp + c; }
};
struct PartGaps {
  const uint8_t* base;
  int hpo;
  __device__ __forceinline__ const float* at(int o, int c) const {
    return reinterpret_cast<const float*>(base + ((o * hpo + (c >> 5)) << 8)) + (((c & 31) + 4 * (o & 7)) & 31);
  }
};

// Sum of one output's span partials rr[0 .. C) in an order that depends only on C: eight
// interleaved sequences s_i = rr[i] + rr[i + 8] + ... (each from 0, in index order), then
// ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)).  Q consecutive lanes (1, 2, 4 or 8, aligned
// to Q) share the output: the lane at position sub of its group forms sequences sub, sub + Q, ...
// and the group combines them with shuffles along the same tree (IEEE addition is commutative,
// so both lanes of a pair get the same bits).  Every lane of the warp must call it; the result
// is the same for every Q.
template <int Q, class Part>
__device__ __forceinline__ float sum_spans(const Part& P, int o, int C, int sub) {
  constexpr int NK = 8 / Q;
  float s[NK];
#pragma unroll
  for (int k = 0; k < NK; ++k) s[k] = 0.0f;
  for (int j = 0; j < C; j += 8) {
#pragma unroll
    for (int k = 0; k < NK; ++k) {
      const int i = j + sub + Q * k;
      if (i < C) s[k] += *P.at(o, i);
    }
  }
  if (Q >= 2) {
#pragma unroll
    for (int k = 0; k < NK; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], 1);
  }
  if (Q >= 4) {
#pragma unroll
    for (int k = 0; k < NK; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], 2);
  }
  if (Q == 8) return s[0] + __shfl_xor_sync(0xffffffffu, s[0], 4);
  if (Q == 4) return s[0] + s[1];
  if (Q == 2) return (s[0] + s[1]) + (s[2] + s[3]);
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// The same sum (one lane per output) for R outputs o[r] at once (the eight floats of each group of
// eight spans may be read past C): every load of a group of eight spans is issued before the first
// add, as two 16-byte loads per output, so a pass costs one shared-memory round trip per eight
// spans for all R outputs (the queue is long while the units decode).
template <int R, class Part>
__device__ __forceinline__ void sum_spans_batch(float (&out)[R], const Part& P, const int (&o)[R], int C) {
  float s[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int k = 0; k < 8; ++k) s[r][k] = 0.0f;
  }
  for (int j = 0; j < C; j += 8) {
    float4 v[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      v[r][0] = *reinterpret_cast<const float4*>(P.at(o[r], j));
      v[r][1] = *reinterpret_cast<const float4*>(P.at(o[r], j + 4));
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float w[8] = {v[r][0].x, v[r][0].y, v[r][0].z, v[r][0].w, v[r][1].x, v[r][1].y, v[r][1].z, v[r][1].w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (j + k < C) s[r][k] += w[k];
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
    out[r] = ((s[r][0] + s[r][1]) + (s[r][2] + s[r][3])) + ((s[r][4] + s[r][5]) + (s[r][6] + s[r][7]));
}

// Loads the NSC = max(1, 128 / bs) scales of one span of one row (NSC * ES bytes, aligned to that
// size when K is a multiple of 128) and expands them to one FP32 scale per k block.
template <int KB, bool SC32, int NSC>
__device__ __forceinline__ void span_scales(float (&sk)[kSpanK / KB], uint32_t a) {
  constexpr int NKB = kSpanK / KB;
  constexpr int ES = SC32 ? 4 : 2;
  constexpr int BYTES = NSC * ES;
  uint32_t w[8];
  if (BYTES >= 16) {
#pragma unroll
    for (int q = 0; q < BYTES / 16; ++q) {
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(w[4 * q]), "=r"(w[4 * q + 1]), "=r"(w[4 * q + 2]), "=r"(w[4 * q + 3]) : "r"(a + 16 * q));
    }
  } else if (BYTES == 8) {
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(a));
  } else if (BYTES == 4) {
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[0]) : "r"(a));
  } else {
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
    w[0] = h;
  }
  float v[NSC];
#pragma unroll
  for (int i = 0; i < NSC; ++i) {
    if (SC32) {
      v[i] = __uint_as_float(w[i]);
    } else {
      const uint32_t word = w[i >> 1];
      v[i] = __half2float(__ushort_as_half((unsigned short)((i & 1) ? (word >> 16) : (word & 0xffffu))));
    }
  }
#pragma unroll
  for (int j = 0; j < NKB; ++j) sk[j] = v[j / (NKB / NSC)];
}

// x of one span for this lane: KB / 4 halves per k block (16-byte loads from xg; blocks at or past
// nkb are zero unless the span is full).
template <int KB, bool FULL>
__device__ __forceinline__ void load_span_x(uint32_t (&xr)[kSpanK / KB][KB / 8], const uint8_t* xg, int nkb) {
#pragma unroll
  for (int j = 0; j < kSpanK / KB; ++j) {
#pragma unroll
    for (int q = 0; q < KB / 32; ++q) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (FULL || j < nkb) v = ld_x_v4(xg + j * (KB * 2) + 16 * q);
      xr[j][4 * q + 0] = v.x; xr[j][4 * q + 1] = v.y; xr[j][4 * q + 2] = v.z; xr[j][4 * q + 3] = v.w;
    }
  }
}

// d = A * B (the accumulator input is zero).
__device__ __forceinline__ void mma16816_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// One unit: 16 weight rows x one span (128 k) of a tile.  b0, b1: shared address of the span's row
// of MMA row g and of MMA row g + 8 (row starts, multiples of 128) plus 64 when the span is the
// second half of its box; the lane's bytes of k block j sit at b0 ^ off0[j] and b1 ^ off1[j]
// (off < 128 holds the lane's byte offset and the row's swizzle).  s0a, s1a: the two rows' scale
// rows (at the span's first scale).  xr: this lane's x of the span (load_span_x; lanes whose batch
// row g is at or above the batch hold the last batch row: their MMA columns are never stored).
// NSC > 0: the span is full and its NSC scales per row are one aligned vector (K a multiple of
// 128); NSC == 0: the general case, nkb k blocks present, scale index of block j = sidx0 +
// (j >> sshift) relative to s0a / s1a.  MMA rows past the tile hold whatever the ring holds there;
// rows are independent in the MMA and those results are never stored.
// KB = 64: per 64-k block, 8 packed bytes per lane per row and 4 MMAs; KB = 32: 4 bytes, 2 MMAs.
// acc[0], acc[1]: MMA row g, batch rows 2t, 2t + 1; acc[2], acc[3]: MMA row g + 8.
template <int KB, bool SC32, int NSC, bool WIDE>
__device__ __forceinline__ void mma_unit(float (&acc)[4], uint32_t b0, uint32_t b1, const uint32_t (&off0)[kSpanK / KB],
                                         const uint32_t (&off1)[kSpanK / KB], uint32_t s0a, uint32_t s1a,
                                         const uint32_t (&xr)[kSpanK / KB][KB / 8], int sidx0, int sshift, int nkb,
                                         uint32_t lut, int lane) {
  constexpr int NKB = kSpanK / KB;     // k blocks per full span
  constexpr int RUN = KB / 8;          // packed bytes per lane per row per k block
  constexpr int NMMA = KB / 16;        // MMAs per k block
  constexpr bool FULL = NSC > 0;
  constexpr int ES = SC32 ? 4 : 2;
  const int t = lane & 3;
  // packed bytes of both rows, per k block
  uint32_t w0[NKB][RUN / 4], w1[NKB][RUN / 4];
#pragma unroll
  for (int j = 0; j < NKB; ++j) {
    if (FULL || j < nkb) {
      if (RUN == 8) {
        const uint2 p = lds_ring64(b0 ^ off0[j]), q = lds_ring64(b1 ^ off1[j]);
        w0[j][0] = p.x; w0[j][RUN / 4 - 1] = p.y;
        w1[j][0] = q.x; w1[j][RUN / 4 - 1] = q.y;
      } else {
        w0[j][0] = lds_ring32(b0 ^ off0[j]);
        w1[j][0] = lds_ring32(b1 ^ off1[j]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < RUN / 4; ++i) w0[j][i] = w1[j][i] = 0u;
    }
  }
  // one scale per k block and row
  float sk0[NKB], sk1[NKB];
  if (FULL) {
    span_scales<KB, SC32, (NSC > 0 ? NSC : 1)>(sk0, s0a);
    span_scales<KB, SC32, (NSC > 0 ? NSC : 1)>(sk1, s1a);
  } else {
    // lane t loads blocks j = t, t + 4 for both rows; shuffled per block
    constexpr int NH = (NKB + 3) / 4;
    float sv0[NH], sv1[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const int j = t + 4 * h;
      float a = 0.0f, b = 0.0f;
      if (j < nkb) {
        const uint32_t off = (uint32_t)((sidx0 + (j >> sshift)) * ES);
        a = SC32 ? lds_scale32(s0a + off) : lds_scale16(s0a + off);
        b = SC32 ? lds_scale32(s1a + off) : lds_scale16(s1a + off);
      }
      sv0[h] = a;
      sv1[h] = b;
    }
#pragma unroll
    for (int j = 0; j < NKB; ++j) {
      sk0[j] = __shfl_sync(0xffffffffu, sv0[j / 4], (lane & ~3) | (j & 3));
      sk1[j] = __shfl_sync(0xffffffffu, sv1[j / 4], (lane & ~3) | (j & 3));
    }
  }
#pragma unroll
  for (int j = 0; j < NKB; ++j) {
    if (FULL || j < nkb) {
      float d[4];
#pragma unroll
      for (int s = 0; s < NMMA; ++s) {
        // slot t: packed byte 2s of the lane's run (k 4s, 4s + 1); slot t + 4: byte 2s + 1
        const uint32_t ww0 = w0[j][(2 * s) >> 2], ww1 = w1[j][(2 * s) >> 2];
        const int b = (2 * s) & 3;
        const uint32_t l4 = (uint32_t)lane * 4u;
        const uint32_t a[4] = {lut_pair<WIDE>(lut, l4, ww0, b), lut_pair<WIDE>(lut, l4, ww1, b),
                               lut_pair<WIDE>(lut, l4, ww0, b + 1), lut_pair<WIDE>(lut, l4, ww1, b + 1)};
        if (s == 0) mma16816_first(d, a, xr[j][2 * s], xr[j][2 * s + 1]);
        else mma16816(d, a, xr[j][2 * s], xr[j][2 * s + 1]);
      }
      acc[0] = fmaf(sk0[j], d[0], acc[0]);
      acc[1] = fmaf(sk0[j], d[1], acc[1]);
      acc[2] = fmaf(sk1[j], d[2], acc[2]);
      acc[3] = fmaf(sk1[j], d[3], acc[3]);
    }
  }
}

}  // namespace w4
