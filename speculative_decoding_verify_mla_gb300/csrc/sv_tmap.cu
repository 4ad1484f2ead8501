// sv_tmap.cu - TMA tensor-map encoding for the launchers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "sv_host.h"

namespace sv {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                int rank, const cuuint64_t* dims, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle) {
  auto encode = get_encode_fn();
  if (!encode || rank < 1 || rank > 5) return false;
  cuuint64_t strides[4];
  cuuint64_t acc = (cuuint64_t)elem_bytes;
  for (int d = 0; d + 1 < rank; ++d) {
    acc *= dims[d];
    strides[d] = acc;
  }
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return encode(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sv
