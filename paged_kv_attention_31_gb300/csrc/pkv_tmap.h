// pkv_tmap.h -- host-side TMA tensor-map encoding shared by the kernels that
// fetch pool pages with cp.async.bulk.tensor.  The driver entry point is
// resolved through the runtime, so the library does not link libcuda.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace pkv {

// Resolved once per process (a function-local static: thread-safe
// initialisation); null if the driver does not provide the entry point.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 4-D tiled map (128-byte swizzle unless told otherwise): dims (inner first)
// d0..d3, byte strides of d1..d3, box b0..b3, elements of `type`.
inline bool make_map_4d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t d0,
                        uint64_t d1, uint64_t d2, uint64_t d3, uint64_t s1, uint64_t s2,
                        uint64_t s3, uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {s1, s2, s3};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, type, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv
