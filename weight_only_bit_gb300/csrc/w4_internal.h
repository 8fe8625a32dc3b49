// w4_internal.h -- host-side declarations shared by libw4's translation units (not installed).
#pragma once
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace w4 {

// Increments the process-wide count of kernel launches issued by the library.
void note_launch();

// Test hook: returns 1 once (and clears the request) after w4_inject_timeout_once() was called.
int take_fault_injection();

cudaError_t launch_quantize_nf4(const float* W, uint8_t* packed, float* absmax, const float* codebook,
                                int N, int K, int bs, cudaStream_t stream);
cudaError_t launch_quantize_int4(const float* W, uint8_t* packed, __half* scale, int N, int K, int gs,
                                 cudaStream_t stream);
cudaError_t launch_quantize_fp4(const float* W, uint8_t* packed, __half* scale, int N, int K, int gs,
                                cudaStream_t stream);
cudaError_t launch_dequantize_fp4(const uint8_t* packed, const __half* scale, float* out, int N, int K, int gs,
                                  cudaStream_t stream);
cudaError_t launch_dequantize_nf4(const uint8_t* packed, const float* absmax, const float* codebook,
                                  float* out, int N, int K, int bs, cudaStream_t stream);
cudaError_t launch_dequantize_int4(const uint8_t* packed, const __half* scale, float* out, int N, int K,
                                   int gs, cudaStream_t stream);

// One GEMV on CUDA cores (batches 1 ... 8 per launch; the caller splits larger batches).  Returns
// cudaErrorNotSupported for shapes the kernel does not serve.
cudaError_t launch_gemv_simt(int format, const uint8_t* packed, const void* scales, const float* codebook,
                             const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                             cudaStream_t stream);

// Launch geometry of the tcgen05 GEMV (host only): MMA batch columns, packed slots, x / A stages,
// CTAs per cluster along K (1: persistent over row tiles), CTAs, threads, dynamic shared memory.
struct Tc5Plan {
  int nb, np, ns, ks, grid, threads, smem;
};
bool plan_tc5(int M, int N, int K, int bs, int sms, Tc5Plan* out);

// CUDA-core launches of a batch-M GEMV (host only): rows of the widest launch, launches, and that
// launch's threads, dynamic shared memory and ring stages.  False if the shape is unsupported.
struct SimtPlan {
  int mb, launches, threads, smem, stages;
};
bool plan_simt(int format, int M, int K, int bs, SimtPlan* out);

// One GEMV on the 5th-generation tensor cores (tcgen05, batch 1 ... 128; used from batch 9).
// cudaErrorNotSupported when the shape is not one it takes (K % 64 != 0, unaligned bases).
cudaError_t launch_gemv_tc5(int format, const uint8_t* packed, const void* scales, const float* codebook,
                            const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                            cudaStream_t stream);

// One GEMV on the tensor cores with mma.sync (batch 32 ... 128).
cudaError_t launch_gemv_tc(int format, const uint8_t* packed, const void* scales, const float* codebook,
                           const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                           cudaStream_t stream);

// Largest batch (8, 4, 2 or 1) one CUDA-core launch serves for this format, K and block size
// (0 if none: the shape is unsupported).
int simt_max_batch(int format, int K, int bs);

int device_sm_count();

// 2-D tiled TMA map over a row-major [rows][cols] array of 1-byte (es = 1) or FP16 (es = 2) elements:
// box of box_cols x box_rows, 128-byte swizzle, zeros outside the array.  False if the driver
// cannot encode it (base not 16-byte aligned, row bytes not a multiple of 16, ...).
bool encode_tmap_2d(CUtensorMap* m, int es, const void* base, long long cols, long long rows, int box_cols,
                    int box_rows);

// Unique id of the CUDA context current on this thread (the runtime's primary context of the current
// device; a new id after cudaDeviceReset), or 0 if the driver cannot say.
unsigned long long current_context_id();

// One-time set-up of a kernel's attributes (shared-memory size and the like), repeated for each
// device and again if that device's context changes (attributes do not survive cudaDeviceReset).
// One instance per kernel instantiation.
struct FuncAttrCache {
  static constexpr int kDevices = 64;
  std::mutex mu;
  unsigned long long ctx[kDevices] = {};
  template <class F>
  cudaError_t ensure(F&& set_attrs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
    const unsigned long long c = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (c != 0 && ctx[dev] == c) return cudaSuccess;
    const cudaError_t e = set_attrs();
    if (e == cudaSuccess) ctx[dev] = c;
    return e;
  }
};

// Each translation unit's device error word (see w4_common.cuh), read and cleared on the current
// device: the CUDA-core kernels' and the tcgen05 kernel's.
unsigned int read_clear_error_persist();
unsigned int read_clear_error_tc5();

// A whole decode step in one persistent launch of the batch 1 ... 8 kernel.  GEMVs are grouped into
// levels (0, 1, ... non-decreasing along the array); a level reads its x only after every GEMV of
// the previous level is complete.  counters: device memory of (number of levels + 1) words, zero
// before the first launch; the kernel leaves it zero again.  Tables: device memory of
// step_tables_bytes(n) bytes, 128-byte aligned, holding what step_simt_tables() builds for the
// same arguments and that base address (tensor maps, levels, GEMVs); written once, read by every
// launch.
constexpr int kStepMaxGemvs = 256;
struct StepJob {
  const uint8_t* packed;
  const void* scales;
  const __half* x;
  __half* y;
  int N, K, bs, level;
};
size_t step_tables_bytes(int n);
cudaError_t step_simt_tables(int format, const StepJob* jobs, int n, int M, const void* dev_base, void* blob);
cudaError_t launch_step_simt(int format, const StepJob* jobs, int n, int M, const float* codebook, unsigned* counters,
                             const void* dev_tables, bool pdl, cudaStream_t stream);

// The same launch with the level counters and the tables in fixed arrays inside the library (no
// caller memory): the tables are copied in on `stream` before the launch.
int noalloc_max_levels();
cudaError_t launch_step_simt_noalloc(int format, const StepJob* jobs, int n, int M, const float* codebook,
                                     int nlevels, cudaStream_t stream);

}  // namespace w4
