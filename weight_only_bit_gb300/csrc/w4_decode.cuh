// w4_decode.cuh -- on-chip decoding of packed 4-bit weights against x held in registers.
//
// One "chunk" is 16 packed bytes = 32 consecutive weights of one row.  A consumer thread owns one
// chunk position of x and multiplies it with that chunk of many rows.
//
//   NF4 ("LLM Quantization on RTX 4060", sections "Standard Expectation from Quantization" and
//   "Kernel Implementation"): a 256-entry table indexed by a whole packed byte returns both code
//   values (FP16) as one half2, element 2j in the low half; one copy of the table per lane, entry b
//   of lane l at word b * 32 + l, so any pattern of bytes across a warp is conflict-free.  Products
//   FP16 x FP16 are exact in FP32 (mixed-precision FMA), sums are FP32, and the block's FP32 absmax
//   multiplies the chunk's partial sum.
//
//   INT4 ("My Triton Kernel Ties bitsandbytes", section "The kernels"): w_hat = (q - 8) * s.  x is
//   converted once to 16-bit fixed point with one exponent per chunk, X = x * 2^(15 - E) where
//   max |x| < 2^E (exact for every |x| >= 2^(E-5)), and split into a signed high byte and an
//   unsigned low byte; dp4a multiplies four nibbles (isolated as bytes) with four digits, so
//   sum (q - 8) x = 2^(E-15) * (256 sum q Xh + sum q Xl - 8 sum X), scaled by s.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "w4_common.cuh"

namespace w4 {

constexpr int kLutBytes = 256 * 32 * 4;   // NF4 byte-pair table, one copy per lane

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

// x: a plain (weak, L1-cached) load.  x may have been written by another SM earlier in the same
// launch; the reader's CTA acquired that writer's release before any thread loads x, which makes
// the write visible to these loads.  Every thread of a CTA reads its slice directly: L1 merges the
// copies that threads sharing a chunk request, so L2 sees each line about once per SM.
__device__ __forceinline__ uint4 ld_x_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// acc += lo(c) * lo(x) + hi(c) * hi(x); products exact (FP16 x FP16 fits FP32), FP32 sums.
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

// Builds the NF4 byte-pair table: entry b = half2(fp16(code[b >> 4]), fp16(code[b & 15])),
// replicated for every lane.  Called by `nthreads` threads numbered t.
__device__ __forceinline__ void build_nf4_lut(uint32_t* lut, const float* __restrict__ codebook, int t, int nthreads) {
  for (int i = t; i < 256 * 32; i += nthreads) {
    const int b = i >> 5;
    const __half lo = __float2half_rn(__ldg(codebook + (b >> 4)));
    const __half hi = __float2half_rn(__ldg(codebook + (b & 15)));
    lut[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
}

// x of one chunk, for MB batch rows.  NF4: 16 half2 pairs per row.  INT4: 16 digit words per row
// (for packed word i: high and low bytes of X at elements 8i+1,3,5,7 -- the low nibbles -- then at
// 8i+0,2,4,6 -- the high nibbles), plus the chunk factor 2^(E-15) and 8 * sum X.
template <int FMT, int MB>
struct XSlice {
  uint32_t v[MB][16];
  float f[MB];
  int s8[MB];
};

// Loads the slice of x at `chunk` (32 elements) for batch rows m < M (zeros above M); x is row-major
// [M][K] in global memory.
template <int FMT, int MB>
__device__ __forceinline__ void load_x_slice(XSlice<FMT, MB>& xs, const __half* __restrict__ x, int M, int K,
                                             int chunk) {
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    uint32_t h[16];
    if (m < M) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(x + (size_t)m * K + (size_t)chunk * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = ld_x_v4(src + 16 * i);
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
      // E: mx < 2^E with mx = max |x| (frexp's exponent; E = 0 for mx = 0), from the FP32 bits
      __half2 amax = __habs2(*reinterpret_cast<const __half2*>(&h[0]));
#pragma unroll
      for (int i = 1; i < 16; ++i) amax = __hmax2(amax, __habs2(*reinterpret_cast<const __half2*>(&h[i])));
      const float mx = fmaxf(__low2float(amax), __high2float(amax));
      const int E = mx > 0.0f ? (int)(__float_as_uint(mx) >> 23) - 126 : 0;
      const float up = __uint_as_float((uint32_t)(127 + 15 - E) << 23);   // 2^(15 - E)
      // X = rint(x * 2^(15-E)): the product is exact, and adding 1.5 * 2^23 in the same FMA rounds
      // it to the nearest integer (ties to even), left in the low mantissa bits
      int X[32];
      int sx = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
        X[2 * i] = (int)(__float_as_uint(fmaf(f2.x, up, 12582912.0f)) - 0x4B400000u);
        X[2 * i + 1] = (int)(__float_as_uint(fmaf(f2.y, up, 12582912.0f)) - 0x4B400000u);
        sx += X[2 * i] + X[2 * i + 1];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // 16-bit pairs, then the high and low bytes of four odd (low-nibble) and four even elements
        uint32_t po01, po23, pe01, pe23;
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(po01) : "r"(X[8 * i + 1]), "r"(X[8 * i + 3]));
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(po23) : "r"(X[8 * i + 5]), "r"(X[8 * i + 7]));
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(pe01) : "r"(X[8 * i + 0]), "r"(X[8 * i + 2]));
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(pe23) : "r"(X[8 * i + 4]), "r"(X[8 * i + 6]));
        asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(xs.v[m][4 * i + 0]) : "r"(po01), "r"(po23));
        asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(xs.v[m][4 * i + 1]) : "r"(po01), "r"(po23));
        asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(xs.v[m][4 * i + 2]) : "r"(pe01), "r"(pe23));
        asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(xs.v[m][4 * i + 3]) : "r"(pe01), "r"(pe23));
      }
      xs.f[m] = __uint_as_float((uint32_t)(127 + E - 15) << 23);       // 2^(E - 15)
      xs.s8[m] = 8 * sx;
    }
  }
}

// INT4 digit table shared by the threads of a CTA: for chunk c of batch row m, its 16 digit words,
// the factor and 8 * sum X at word (m * kXDigitWords + w) * cpr + c (a warp's accesses to one word
// are contiguous: no bank conflict).
constexpr int kXDigitWords = 18;

template <int MB>
__device__ __forceinline__ void put_x_digits(uint32_t* xd, const XSlice<1, MB>& xs, int M, int cpr, int chunk) {
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m < M) {
#pragma unroll
      for (int w = 0; w < 16; ++w) xd[(m * kXDigitWords + w) * cpr + chunk] = xs.v[m][w];
      xd[(m * kXDigitWords + 16) * cpr + chunk] = __float_as_uint(xs.f[m]);
      xd[(m * kXDigitWords + 17) * cpr + chunk] = (uint32_t)xs.s8[m];
    }
  }
}

template <int MB>
__device__ __forceinline__ void get_x_digits(XSlice<1, MB>& xs, const uint32_t* xd, int M, int cpr, int chunk) {
#pragma unroll
  for (int m = 0; m < MB; ++m) {
    if (m < M) {
#pragma unroll
      for (int w = 0; w < 16; ++w) xs.v[m][w] = xd[(m * kXDigitWords + w) * cpr + chunk];
      xs.f[m] = __uint_as_float(xd[(m * kXDigitWords + 16) * cpr + chunk]);
      xs.s8[m] = (int)xd[(m * kXDigitWords + 17) * cpr + chunk];
    } else {
#pragma unroll
      for (int w = 0; w < 16; ++w) xs.v[m][w] = 0u;
      xs.f[m] = 1.0f;
      xs.s8[m] = 0;
    }
  }
}

// One chunk of R rows (R = 1 or 2, decoded together so their shared-memory reads overlap):
// part[r][m] = sum over the chunk's 32 weights of w_hat[r] * x[m].  wv[r]: the chunk's 16 packed
// bytes of row r; scale_addr[r]: shared-memory address of row r's scale for the chunk (FP32 absmax
// for NF4, FP16 s for INT4); lut_lane: this lane's table base (NF4).
template <int FMT, int MB, int R>
__device__ __forceinline__ void chunk_dot(float (&part)[R][MB], const uint4 (&wv)[R], const uint32_t (&scale_addr)[R],
                                          uint32_t lut_lane, const XSlice<FMT, MB>& xs) {
  if (FMT == 0) {
    float a[R];
#pragma unroll
    for (int r = 0; r < R; ++r) a[r] = __uint_as_float(lds32(scale_addr[r]));
    constexpr int NA = MB >= 4 ? 1 : 4 / MB;   // independent accumulators per (row, batch row)
    float acc[R][MB][NA];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int q = 0; q < NA; ++q) acc[r][m][q] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t c2[R][4];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t w = i == 0 ? wv[r].x : i == 1 ? wv[r].y : i == 2 ? wv[r].z : wv[r].w;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t byte;
          asm("prmt.b32 %0, %1, 0, %2;" : "=r"(byte) : "r"(w), "r"(0x4440 + b));
          c2[r][b] = lds32(lut_lane + byte * 128u);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int m = 0; m < MB; ++m) mixed_dot2(acc[r][m][(4 * i + b) % NA], c2[r][b], xs.v[m][4 * i + b]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < NA; ++q) sum += acc[r][m][q];
        part[r][m] = sum * a[r];
      }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float s = __half2float(__ushort_as_half((unsigned short)lds_u16(scale_addr[r])));
      const uint32_t w4[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
      int ah[MB], al[MB];
#pragma unroll
      for (int m = 0; m < MB; ++m) { ah[m] = 0; al[m] = 0; }
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
        part[r][m] = (float)tot * (s * xs.f[m]);
      }
    }
  }
}

}  // namespace w4
