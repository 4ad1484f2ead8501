// sv_host.h - host-side helpers shared by the kernels' launchers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

namespace sv {

// cuTensorMapEncodeTiled from the driver (through the runtime's entry-point
// query, so the library does not link libcuda); nullptr when unavailable.
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn();

// Tiled tensor map (128-byte swizzle unless stated) over a row-major tensor
// (dims[0] is the innermost, contiguous dimension; rank <= 5).  False on
// failure.
bool encode_map(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                int rank, const cuuint64_t* dims, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

}  // namespace sv
