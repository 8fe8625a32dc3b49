// w4_tc.cu -- fused 4-bit dequant-GEMM on the tensor cores for batches 32 ... 128 (sm_103a).
//
// At these batches every decoded weight feeds 32-128 multiply-adds, so the work is a dense
// contraction and belongs on the tensor cores; at batch 1 it is not ("My Triton Kernel Ties
// bitsandbytes", section "Why Marlin is still faster": a tl.dot rewrite at batch 1 was 4-7x
// slower).  Weights are still decoded on chip and never written back ("LLM Quantization on RTX
// 4060", section "Fused Kernel: Moving Dequantization On-Chip"); the batch-dependent switch of
// paths is the one "Do Quantization and Sparsity make LLM Inference Faster ?" describes for
// bitsandbytes (section "NF4: fast at batch 1, slower at larger batches"), without the
// out-of-place dequantisation.
//
// y^T[N][M] = W_hat[N][K] . x^T[K][M] with mma.sync.m16n8k16 (FP16 x FP16 -> FP32):
//   * A = weights.  Warp w of a CTA owns 16 rows.  A packed byte holds the element pair (2j, 2j+1)
//     of one row, which is exactly one A-fragment register (two consecutive k of one row), so the
//     byte-pair table of w4_decode.cuh (NF4 code values, q - 8 for INT4, E2M1 values for FP4) yields
//     fragments
//     directly; the block scale (FP32 absmax rounded to FP16, or the FP16 INT4 / FP4 scale) multiplies
//     each fragment (one HMUL2 per two weights).
//   * K is reordered identically for A and B: in each 64-k chunk, thread t (= lane % 4) owns the
//     8 consecutive packed bytes 8t ... 8t+7 of its two rows (one 8-byte load each); in k-step s
//     its fragment slots t and t+4 take element pairs 8t+2s and 8t+2s+1.  The B fragment then
//     reads x elements 16t+4s ... 16t+4s+3: one 8-byte shared-memory load.
//   * B = x, staged per 256-k window in shared memory (double-buffered, rows padded).
//   * Split-K: the K windows are divided among the CTAs of a thread-block cluster; each CTA
//     leaves its FP32 partial tile in its shared memory, and after a cluster barrier CTA r sums
//     rows [r*128/ks, (r+1)*128/ks) over the cluster in rank order through distributed shared
//     memory and writes y.  No global scratch; results do not depend on timing.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4_common.cuh"
#include "w4_decode.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr int kTcWarps = 8;
constexpr int kTcRows = kTcWarps * 16;     // weight rows per CTA
constexpr int kTcWin = 256;                // k per window
constexpr int kTcXPad = 8;                 // halves of padding per staged x row

struct TcParams {
  const uint8_t* packed;
  const void* scales;
  const float* codebook;
  const __half* x;
  __half* y;
  int M, N, K, bs;
  int ks;            // CTAs per cluster along K
  int nwin;          // windows of kTcWin along K (the last may be shorter)
};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load a float from the shared memory of CTA `rank` of this cluster (after a cluster barrier, so
// the value is stable and the loads may be issued together).
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}

// 16-byte asynchronous copy global -> shared (through L2 only), completion by commit groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Scale of row `row` for the block holding k index `k`, as a half2 of two equal values.
template <int FMT>
__device__ __forceinline__ uint32_t tc_scale2(const void* scales, int row, int k, int K, int bs) {
  __half s;
  if (FMT == 0) {
    s = __float2half_rn(__ldg(reinterpret_cast<const float*>(scales) + (size_t)row * (K / bs) + k / bs));
  } else {
    s = reinterpret_cast<const __half*>(scales)[(size_t)row * (K / bs) + k / bs];
  }
  const uint32_t h = __half_as_ushort(s);
  return h | (h << 16);
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kTcWarps * 32, NT >= 16 ? 1 : 2) w4_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int XS = kTcWin + kTcXPad;                  // staged x row stride (halves)
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem);    // byte-pair table, one copy per lane
  __half* xbuf = reinterpret_cast<__half*>(smem + kLutBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;          // fragment row group
  const int t = lane & 3;           // fragment thread-in-group
  const uint32_t rank = cluster_ctarank();
  const int rb = blockIdx.x / p.ks;                     // row block
  const int row0 = rb * kTcRows + warp * 16;
  const int rA = row0 + g, rB = row0 + g + 8;           // this thread's two rows
  const bool okA = rA < p.N, okB = rB < p.N;
  const int M = p.M;

  // decode table: NF4 code values, q - 8 for INT4, E2M1 values for FP4
  build_lut(lut, FMT, p.codebook, (int)threadIdx.x, (int)blockDim.x);
  const uint32_t lut_lane = smem_u32(lut) + (uint32_t)lane * 4u;
  pdl_launch_dependents();
  pdl_wait();

  // this CTA's windows along K
  const int w0 = (int)((long long)rank * p.nwin / p.ks);
  const int w1 = (int)((long long)(rank + 1) * p.nwin / p.ks);

  float acc[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;

  const uint8_t* rowA = p.packed + (size_t)(okA ? rA : 0) * (p.K / 2);
  const uint8_t* rowB = p.packed + (size_t)(okB ? rB : 0) * (p.K / 2);

  // stage window w of x into buffer b: rows n < M, zero rows up to NT * 8
  auto stage_x = [&](int w, int b) {
    __half* xb = xbuf + (size_t)b * (NT * 8) * XS;
    const int k0 = w * kTcWin;
    const int kw = min(kTcWin, p.K - k0);
    const int units = NT * 8 * (kTcWin / 8);           // 16-byte units of the padded-free area
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int n = u / (kTcWin / 8);
      const int c = (u - n * (kTcWin / 8)) * 8;
      if (n < M && c < kw) {
        cp_async16(xb + (size_t)n * XS + c, p.x + (size_t)n * p.K + k0 + c);
      } else {
        *reinterpret_cast<uint4*>(xb + (size_t)n * XS + c) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };

  // packed bytes and scales of one window for this thread's two rows (loaded one window ahead)
  struct Win {
    uint2 a[4], b[4];
    uint32_t sa[4], sb[4];
  };
  auto load_win = [&](int w, Win& v) {
    const int k0 = w * kTcWin;
    const int nch = min(kTcWin, p.K - k0) / 64;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int kc = k0 + 64 * c;
      v.a[c] = make_uint2(0, 0); v.b[c] = make_uint2(0, 0); v.sa[c] = 0u; v.sb[c] = 0u;
      if (c < nch) {
        if (okA) {
          v.a[c] = *reinterpret_cast<const uint2*>(rowA + kc / 2 + 8 * t);
          v.sa[c] = tc_scale2<FMT>(p.scales, rA, kc + 16 * t, p.K, p.bs);
        }
        if (okB) {
          v.b[c] = *reinterpret_cast<const uint2*>(rowB + kc / 2 + 8 * t);
          v.sb[c] = tc_scale2<FMT>(p.scales, rB, kc + 16 * t, p.K, p.bs);
        }
      }
    }
  };

  Win cur, nxt;
  if (w0 < w1) {
    load_win(w0, cur);
    stage_x(w0, 0);
  }
  cp_async_wait_all();
  __syncthreads();
  for (int w = w0; w < w1; ++w) {
    const int b = (w - w0) & 1;
    if (w + 1 < w1) {
      load_win(w + 1, nxt);                             // weights of the next window in flight
      stage_x(w + 1, b ^ 1);                            // and its x
    }
    const int k0 = w * kTcWin;
    const int nchunk = min(kTcWin, p.K - k0) / 64;
    const __half* xb = xbuf + (size_t)b * (NT * 8) * XS;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c >= nchunk) break;
      uint32_t fa[8], fb[8];                            // 8 element pairs of each row, scaled
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t wa = i < 4 ? cur.a[c].x : cur.a[c].y, wb = i < 4 ? cur.b[c].x : cur.b[c].y;
        uint32_t ba, bb;
        asm("prmt.b32 %0, %1, 0, %2;" : "=r"(ba) : "r"(wa), "r"(0x4440 + (i & 3)));
        asm("prmt.b32 %0, %1, 0, %2;" : "=r"(bb) : "r"(wb), "r"(0x4440 + (i & 3)));
        const uint32_t ca = lds32(lut_lane + ba * 128u), cb = lds32(lut_lane + bb * 128u);
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(fa[i]) : "r"(ca), "r"(cur.sa[c]));
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(fb[i]) : "r"(cb), "r"(cur.sb[c]));
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t a[4] = {fa[2 * s], fb[2 * s], fa[2 * s + 1], fb[2 * s + 1]};
        const int kx = 64 * c + 16 * t + 4 * s;         // k offset in the window of this thread's B pair
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const uint2 bv = *reinterpret_cast<const uint2*>(xb + (size_t)(8 * j + g) * XS + kx);
          mma16816(acc[j], a, bv.x, bv.y);
        }
      }
    }
    if (w + 1 < w1) cur = nxt;
    cp_async_wait_all();                               // this thread's copies of the next window
    __syncthreads();                                   // window b consumed, next staged
  }

  // partial tile into this CTA's shared memory: part[row][n], FP32
  float* part = reinterpret_cast<float*>(smem + kLutBytes);
  const int PS = NT * 8 + 1;                           // odd row stride
  __syncthreads();
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int n = 8 * j + 2 * t;
    const int lr = warp * 16 + g;
    part[lr * PS + n] = acc[j][0];
    part[lr * PS + n + 1] = acc[j][1];
    part[(lr + 8) * PS + n] = acc[j][2];
    part[(lr + 8) * PS + n + 1] = acc[j][3];
  }
  cluster_sync();
  // CTA `rank` reduces its share of the rows over the cluster, in rank order
  const int rows_per = (kTcRows + p.ks - 1) / p.ks;
  const int lr0 = rank * rows_per;
  const int lr1 = min(kTcRows, lr0 + rows_per);
  for (int e = threadIdx.x; e < (lr1 - lr0) * M; e += blockDim.x) {
    const int lr = lr0 + e / M;
    const int n = e - (e / M) * M;
    float pv[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) pv[r] = r < p.ks ? ld_dsmem_f32(part + lr * PS + n, (uint32_t)r) : 0.0f;
    float v = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r) v += pv[r];               // rank order
    const int row = rb * kTcRows + lr;
    if (row < p.N) p.y[(size_t)n * p.N + row] = __float2half_rn(v);
  }
  cluster_sync();                                      // keep shared memory alive for the readers
}

template <int FMT, int NT>
static cudaError_t launch_tc_nt(const TcParams& p0, bool pdl, cudaStream_t stream) {
  TcParams p = p0;
  auto kern = w4_tc_kernel<FMT, NT>;
  constexpr int XS = kTcWin + kTcXPad;
  const size_t xbytes = 2 * (size_t)(NT * 8) * XS * sizeof(__half);
  const size_t pbytes = (size_t)kTcRows * (NT * 8 + 1) * sizeof(float);
  const size_t smem = kLutBytes + (xbytes > pbytes ? xbytes : pbytes);
  static FuncAttrCache attrs;
  cudaError_t ea = attrs.ensure([&] {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int nrb = (p.N + kTcRows - 1) / kTcRows;
  // K split: enough CTAs to cover the SMs, at most 8 (a portable cluster) and one window each
  int ks = (device_sm_count() + nrb - 1) / nrb;
  if (ks > 8) ks = 8;
  if (ks > p.nwin) ks = p.nwin;
  if (ks < 1) ks = 1;
  p.ks = ks;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nrb * ks));
  cfg.blockDim = dim3(kTcWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  return e;
}

cudaError_t launch_gemv_tc(int format, const uint8_t* packed, const void* scales, const float* codebook,
                           const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                           cudaStream_t stream) {
  if (M < 32 || M > 128 || K % 64 != 0 || bs < 32) return cudaErrorNotSupported;
  TcParams p;
  p.packed = packed; p.scales = scales; p.codebook = codebook; p.x = x; p.y = y;
  p.M = M; p.N = N; p.K = K; p.bs = bs;
  p.ks = 1;
  p.nwin = (K + kTcWin - 1) / kTcWin;
  const int NT = (M + 7) / 8;
  if (format == 0) {
    if (NT <= 4) return launch_tc_nt<0, 4>(p, pdl, stream);
    if (NT <= 8) return launch_tc_nt<0, 8>(p, pdl, stream);
    return launch_tc_nt<0, 16>(p, pdl, stream);
  }
  if (format == 1) {
    if (NT <= 4) return launch_tc_nt<1, 4>(p, pdl, stream);
    if (NT <= 8) return launch_tc_nt<1, 8>(p, pdl, stream);
    return launch_tc_nt<1, 16>(p, pdl, stream);
  }
  if (NT <= 4) return launch_tc_nt<2, 4>(p, pdl, stream);
  if (NT <= 8) return launch_tc_nt<2, 8>(p, pdl, stream);
  return launch_tc_nt<2, 16>(p, pdl, stream);
}

}  // namespace w4
