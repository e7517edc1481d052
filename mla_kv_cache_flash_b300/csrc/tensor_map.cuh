// Host-side TMA descriptor encoding (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mlakv {

// dims[0] is the contiguous dimension; strides_bytes[i] is the stride of dims[i+1].
// Zero fill out of bounds. Returns cudaErrorInvalidValue if the driver rejects the map.
MLAKV_HIDDEN cudaError_t encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base,
                                           const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                                           CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo);

}  // namespace mlakv
