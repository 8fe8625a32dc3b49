// w4_tmap.cu -- driver entry points the library uses (looked up through the runtime, so there is no
// link against libcuda): the TMA tensor-map encoder and the current context's id.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "w4_internal.h"

namespace w4 {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no link against libcuda).
static EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}

using CtxCurrentFn = CUresult (*)(CUcontext*);
using CtxIdFn = CUresult (*)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
  static CtxCurrentFn cur = nullptr;
  static CtxIdFn id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      cur = reinterpret_cast<CtxCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      id = reinterpret_cast<CtxIdFn>(f);
  });
  if (!cur || !id) return 0;
  CUcontext c = nullptr;
  unsigned long long v = 0;
  if (cur(&c) != CUDA_SUCCESS || c == nullptr || id(c, &v) != CUDA_SUCCESS) return 0;
  return v;
}

bool encode_tmap_2d(CUtensorMap* m, int es, const void* base, long long cols, long long rows, int box_cols,
                    int box_rows) {
  EncodeFn enc = encoder();
  if (!enc || (es != 1 && es != 2)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(cols * es)};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace w4
