// w4_decode.cuh -- shared pieces of the on-chip decoding of packed 4-bit weights.
//
// The decode is a 256-entry table indexed by a whole packed byte that returns both nibbles' values
// (FP16) as one half2, element 2j in the low half ("LLM Quantization on RTX 4060", section "Kernel
// Implementation": the high nibble of byte j is element 2j); one copy of the table per lane, entry
// b of lane l at word b * 32 + l (or b * 64 + l in the 64 KB layout), so any pattern of bytes
// across a warp is conflict-free.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#include "w4_common.cuh"

namespace w4 {

constexpr int kLutBytes = 256 * 32 * 4;   // byte-pair table, one copy per lane
constexpr int kLutWideBytes = 256 * 64 * 4;   // the same at 256-byte entry stride (build_lut, wide)

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
// the write visible to these loads.  Every lane reads the x elements of its own MMA fragments
// directly; L1 merges the requests of the warps that share them, so L2 sees each line about once
// per SM.
__device__ __forceinline__ uint4 ld_x_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Byte-pair table for the format: entry b = half2(v(b >> 4), v(b & 15)), one copy per lane (entry b
// of lane l at word 32 b + l, so any pattern of bytes across a warp is conflict-free).
//   NF4: v(q) = fp16(code[q]);  INT4: v(q) = q - 8;  FP4 (E2M1, sign in bit 3): v(q) = +-{0, 0.5, 1,
//   1.5, 2, 3, 4, 6}[q & 7] ("LLM Compressor 0.14", section "Details worth knowing": the E2M1 grid).
__device__ __forceinline__ float nibble_value(int fmt, const float* __restrict__ codebook, int q) {
  if (fmt == 0) return __ldg(codebook + q);
  if (fmt == 1) return (float)(q - 8);
  // E2M1: exponent e = bits 1-2 (bias 1; e = 0 is subnormal, m / 2), mantissa m = bit 0
  const int mag = q & 7;
  const float v = mag < 2 ? 0.5f * (float)mag : (float)(1 << ((mag >> 1) - 1)) * (mag & 1 ? 1.5f : 1.0f);
  return (q & 8) ? -v : v;
}

// wide = false: entry b of lane l at word 32 b + l (32 KB).  wide = true: at word 64 b + l (64 KB),
// so that entry b of lane l sits at byte 256 b + 4 l, an offset one byte permute forms from the
// packed byte and the lane; words 64 b + 32 ... 64 b + 63 are left free (256 gaps of 128 bytes).
__device__ __forceinline__ void build_lut(uint32_t* lut, int fmt, const float* __restrict__ codebook, int t,
                                          int nthreads, bool wide = false) {
  const int sh = wide ? 6 : 5;
  for (int i = t; i < 256 * 32; i += nthreads) {
    const int b = i >> 5;
    const __half lo = __float2half_rn(nibble_value(fmt, codebook, b >> 4));
    const __half hi = __float2half_rn(nibble_value(fmt, codebook, b & 15));
    lut[(b << sh) + (i & 31)] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
}

}  // namespace w4
