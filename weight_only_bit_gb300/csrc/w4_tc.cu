// w4_tc.cu -- fused 4-bit dequant-GEMM on the tensor cores for batches 32 ... 128 (sm_103a).
// Not built yet in this revision: the dispatcher falls back to CUDA-core launches over batch
// slices of 8 rows when this returns cudaErrorNotSupported.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4_internal.h"

namespace w4 {

cudaError_t launch_gemv_tc(int format, const uint8_t* packed, const void* scales, const float* codebook,
                           const __half* x, __half* y, int M, int N, int K, int bs, bool pdl,
                           cudaStream_t stream) {
  (void)format; (void)packed; (void)scales; (void)codebook; (void)x; (void)y;
  (void)M; (void)N; (void)K; (void)bs; (void)pdl; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace w4
