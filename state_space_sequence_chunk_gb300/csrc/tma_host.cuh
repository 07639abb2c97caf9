// tma_host.cuh -- host-side encoding of TMA tensor maps through the driver's
// cuTensorMapEncodeTiled, fetched at run time from the CUDA runtime so that
// the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

// Encode a tiled map of rank 1..5 (dims[0] contiguous; strides_bytes holds the
// byte strides of dims 1..rank-1).  Returns false if the encoder is unavailable
// or rejects the arguments.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

// Encode a 4-D tiled map.  dims[0] is the contiguous dimension; strides_bytes
// are the byte strides of dims 1..3.  Returns false if the encoder is
// unavailable or rejects the arguments.
bool encode_tmap_4d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    const uint64_t dims[4], const uint64_t strides_bytes[3],
                    const uint32_t box[4], CUtensorMapSwizzle swizzle);

}  // namespace ssd
