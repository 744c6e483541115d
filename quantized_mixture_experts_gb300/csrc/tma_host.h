// Host helpers for TMA tensor maps and device properties.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmoe {

// Encodes a 2-D tiled tensor map: `outer` rows of `inner` elements, rows
// `row_bytes` apart, copied in boxes of box_inner x box_outer elements.
// Returns false when the driver rejects it or the base/stride are not
// 16-byte aligned.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle);

// Encodes a 3-D tiled tensor map: dims[0] innermost (contiguous), dims[1] and
// dims[2] strides_bytes[0] and strides_bytes[1] apart, boxes of box[0..2].
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    const uint64_t dims[3], const uint64_t strides_bytes[2], const uint32_t box[3],
                    CUtensorMapSwizzle swizzle);

// Multiprocessor count of the current device (152 when it cannot be queried).
int device_sm_count();

}  // namespace qmoe
