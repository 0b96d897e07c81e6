// tmap.cu -- TMA tensor maps (cuTensorMapEncodeTiled through the runtime's driver
// entry point, so the library links only the CUDA runtime).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "tmap.h"

namespace spattn {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

}  // namespace

bool make_map(CUtensorMap* map, const void* base, int D, long long rows, long long BH,
              long long dview, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  if (rows < 1) rows = 1;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(D) * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(dview),
                        static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[3] = {row_bytes, row_bytes * static_cast<cuuint64_t>(dview),
                           row_bytes * static_cast<cuuint64_t>(dview) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace spattn
