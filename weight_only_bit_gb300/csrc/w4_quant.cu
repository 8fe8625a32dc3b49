// w4_quant.cu -- NF4 / INT4 / FP4 quantisation and dequantisation kernels (off the decode hot path).
//
// Every rounding decision is the one the C ABI documents, taken in the same precision on every
// run, so the packed codes and scales are reproducible bit for bit:
//   NF4  ("LLM Quantization on RTX 4060: Where 4-bit Decode Falls Behind FP16", sections
//        "Standard Expectation from Quantization" and "Kernel Implementation"):
//        a = max |w| over the block; n = w / a as an IEEE FP32 division (a == 0 -> n = 0);
//        code = number of code-book midpoints (c[i] + c[i+1]) / 2 lying strictly below n,
//        compared exactly in float64 (the nearest code, a tie going to the lower one).
//   INT4 ("My Triton Kernel Ties bitsandbytes", section "The kernels"; "LLM Compressor 0.14",
//        section "Details worth knowing" for rint):
//        s = fp16_rn(fp32(a / 7)); q = clamp(rint(fp32(w / s)), -8, 7) + 8; s == 0 -> q = 8.
//   FP4 E2M1 ("LLM Compressor 0.14", section "Details worth knowing": the grid {0, 0.5, 1, 1.5,
//        2, 3, 4, 6} and its threshold ladder, ties to the even code):
//        s = fp16_rn(fp32(a / 6)); r = fp32(w / s); index = ladder(|r|) over the midpoints of the
//        grid, moving up past an even rung only when |r| > t and past an odd rung when |r| >= t;
//        code = (w < 0) << 3 | index; s == 0 -> code 0.
// Packing: byte j of a row = code(2j) << 4 | code(2j+1).
#include <cstdint>
#include <cuda_fp16.h>

#include "w4_common.cuh"
#include "w4_decode.cuh"
#include "w4_internal.h"

namespace w4 {

// One warp per block of `bs` weights; each lane handles byte pairs j = lane, lane + 32, ...
__global__ void __launch_bounds__(256) quantize_nf4_kernel(const float* __restrict__ W,
                                                           uint8_t* __restrict__ packed,
                                                           float* __restrict__ absmax,
                                                           const float* __restrict__ codebook,
                                                           long long n_blocks, int bs) {
  __shared__ double mid[15];
  if (threadIdx.x < 15) {
    mid[threadIdx.x] = ((double)codebook[threadIdx.x] + (double)codebook[threadIdx.x + 1]) * 0.5;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long blk = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blk >= n_blocks) return;
  const float2* src = reinterpret_cast<const float2*>(W + blk * bs);
  const int pairs = bs >> 1;
  float a = 0.0f;
  for (int j = lane; j < pairs; j += 32) {
    float2 v = src[j];
    a = fmaxf(a, fmaxf(fabsf(v.x), fabsf(v.y)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  uint8_t* dst = packed + blk * pairs;
  for (int j = lane; j < pairs; j += 32) {
    float2 v = src[j];
    uint32_t code[2];
    float e[2] = {v.x, v.y};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const double n = (a > 0.0f) ? (double)__fdiv_rn(e[t], a) : 0.0;
      // count of midpoints strictly below n (binary search over 15 sorted midpoints)
      uint32_t c = 0;
      if (mid[c + 7] < n) c += 8;
      if (mid[c + 3] < n) c += 4;
      if (mid[c + 1] < n) c += 2;
      if (mid[c] < n) c += 1;
      code[t] = c;
    }
    dst[j] = static_cast<uint8_t>((code[0] << 4) | code[1]);
  }
  if (lane == 0) absmax[blk] = a;
}

__global__ void __launch_bounds__(256) quantize_int4_kernel(const float* __restrict__ W,
                                                            uint8_t* __restrict__ packed,
                                                            __half* __restrict__ scale,
                                                            long long n_groups, int gs) {
  const int lane = threadIdx.x & 31;
  const long long grp = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (grp >= n_groups) return;
  const float2* src = reinterpret_cast<const float2*>(W + grp * gs);
  const int pairs = gs >> 1;
  float a = 0.0f;
  for (int j = lane; j < pairs; j += 32) {
    float2 v = src[j];
    a = fmaxf(a, fmaxf(fabsf(v.x), fabsf(v.y)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const __half s16 = __float2half_rn(__fdiv_rn(a, 7.0f));
  const float s = __half2float(s16);
  uint8_t* dst = packed + grp * pairs;
  for (int j = lane; j < pairs; j += 32) {
    float2 v = src[j];
    float e[2] = {v.x, v.y};
    uint32_t q[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float r = (s > 0.0f) ? __fdiv_rn(e[t], s) : 0.0f;
      float ri = rintf(r);
      ri = fminf(fmaxf(ri, -8.0f), 7.0f);
      q[t] = static_cast<uint32_t>(static_cast<int>(ri) + 8);
    }
    dst[j] = static_cast<uint8_t>((q[0] << 4) | q[1]);
  }
  if (lane == 0) scale[grp] = s16;
}

// E2M1 grid index of a magnitude m >= 0 (the threshold ladder; a value on a threshold lands on the
// even index).
__device__ __forceinline__ uint32_t fp4_index(float m) {
  uint32_t i = 0;
  i += m > 0.25f ? 1u : 0u;
  i += m >= 0.75f ? 1u : 0u;
  i += m > 1.25f ? 1u : 0u;
  i += m >= 1.75f ? 1u : 0u;
  i += m > 2.5f ? 1u : 0u;
  i += m >= 3.5f ? 1u : 0u;
  i += m > 5.0f ? 1u : 0u;
  return i;
}

__global__ void __launch_bounds__(256) quantize_fp4_kernel(const float* __restrict__ W,
                                                           uint8_t* __restrict__ packed,
                                                           __half* __restrict__ scale,
                                                           long long n_groups, int gs) {
  const int lane = threadIdx.x & 31;
  const long long grp = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (grp >= n_groups) return;
  const float2* src = reinterpret_cast<const float2*>(W + grp * gs);
  const int pairs = gs >> 1;
  float a = 0.0f;
  for (int j = lane; j < pairs; j += 32) {
    float2 v = src[j];
    a = fmaxf(a, fmaxf(fabsf(v.x), fabsf(v.y)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const __half s16 = __float2half_rn(__fdiv_rn(a, 6.0f));
  const float s = __half2float(s16);
  uint8_t* dst = packed + grp * pairs;
  for (int j = lane; j < pairs; j += 32) {
    float2 v = src[j];
    float e[2] = {v.x, v.y};
    uint32_t q[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float r = (s > 0.0f) ? __fdiv_rn(e[t], s) : 0.0f;
      q[t] = (s > 0.0f && e[t] < 0.0f ? 8u : 0u) | fp4_index(fabsf(r));
    }
    dst[j] = static_cast<uint8_t>((q[0] << 4) | q[1]);
  }
  if (lane == 0) scale[grp] = s16;
}

// Dequantisation: one thread per packed byte (two weights).
__global__ void __launch_bounds__(256) dequantize_nf4_kernel(const uint8_t* __restrict__ packed,
                                                             const float* __restrict__ absmax,
                                                             const float* __restrict__ codebook,
                                                             float* __restrict__ out,
                                                             long long n_bytes, int bs) {
  __shared__ float code[16];
  if (threadIdx.x < 16) code[threadIdx.x] = codebook[threadIdx.x];
  __syncthreads();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_bytes) return;
  const uint32_t b = packed[i];
  const float a = absmax[(2 * i) / bs];   // blocks never straddle rows (K % bs == 0)
  float2 r;
  r.x = __fmul_rn(code[b >> 4], a);
  r.y = __fmul_rn(code[b & 15u], a);
  reinterpret_cast<float2*>(out)[i] = r;
}

__global__ void __launch_bounds__(256) dequantize_int4_kernel(const uint8_t* __restrict__ packed,
                                                              const __half* __restrict__ scale,
                                                              float* __restrict__ out,
                                                              long long n_bytes, int gs) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_bytes) return;
  const uint32_t b = packed[i];
  const float s = __half2float(scale[(2 * i) / gs]);
  float2 r;
  r.x = __fmul_rn(static_cast<float>(static_cast<int>(b >> 4) - 8), s);
  r.y = __fmul_rn(static_cast<float>(static_cast<int>(b & 15u) - 8), s);
  reinterpret_cast<float2*>(out)[i] = r;
}

__global__ void __launch_bounds__(256) dequantize_fp4_kernel(const uint8_t* __restrict__ packed,
                                                             const __half* __restrict__ scale,
                                                             float* __restrict__ out,
                                                             long long n_bytes, int gs) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_bytes) return;
  const uint32_t b = packed[i];
  const float s = __half2float(scale[(2 * i) / gs]);
  float2 r;
  r.x = __fmul_rn(nibble_value(2, nullptr, (int)(b >> 4)), s);
  r.y = __fmul_rn(nibble_value(2, nullptr, (int)(b & 15u)), s);
  reinterpret_cast<float2*>(out)[i] = r;
}

cudaError_t launch_quantize_nf4(const float* W, uint8_t* packed, float* absmax, const float* codebook,
                                int N, int K, int bs, cudaStream_t stream) {
  const long long n_blocks = (long long)N * (K / bs);
  const int warps = 8;
  const long long grid = (n_blocks + warps - 1) / warps;
  quantize_nf4_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(W, packed, absmax, codebook, n_blocks, bs);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_quantize_int4(const float* W, uint8_t* packed, __half* scale, int N, int K, int gs,
                                 cudaStream_t stream) {
  const long long n_groups = (long long)N * (K / gs);
  const int warps = 8;
  const long long grid = (n_groups + warps - 1) / warps;
  quantize_int4_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(W, packed, scale, n_groups, gs);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequantize_nf4(const uint8_t* packed, const float* absmax, const float* codebook,
                                  float* out, int N, int K, int bs, cudaStream_t stream) {
  const long long n_bytes = (long long)N * (K / 2);
  const long long grid = (n_bytes + 255) / 256;
  dequantize_nf4_kernel<<<(unsigned)grid, 256, 0, stream>>>(packed, absmax, codebook, out, n_bytes, bs);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequantize_int4(const uint8_t* packed, const __half* scale, float* out, int N, int K,
                                   int gs, cudaStream_t stream) {
  const long long n_bytes = (long long)N * (K / 2);
  const long long grid = (n_bytes + 255) / 256;
  dequantize_int4_kernel<<<(unsigned)grid, 256, 0, stream>>>(packed, scale, out, n_bytes, gs);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp4(const float* W, uint8_t* packed, __half* scale, int N, int K, int gs,
                                cudaStream_t stream) {
  const long long n_groups = (long long)N * (K / gs);
  const int warps = 8;
  const long long grid = (n_groups + warps - 1) / warps;
  quantize_fp4_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(W, packed, scale, n_groups, gs);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequantize_fp4(const uint8_t* packed, const __half* scale, float* out, int N, int K, int gs,
                                  cudaStream_t stream) {
  const long long n_bytes = (long long)N * (K / 2);
  const long long grid = (n_bytes + 255) / 256;
  dequantize_fp4_kernel<<<(unsigned)grid, 256, 0, stream>>>(packed, scale, out, n_bytes, gs);
  note_launch();
  return cudaGetLastError();
}

}  // namespace w4
