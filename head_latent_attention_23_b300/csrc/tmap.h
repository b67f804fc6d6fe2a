// Host helpers to encode TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point so the library needs no libcuda
// link).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mla {

// Row-major bf16 tensor of `rank` dims (dims[0] innermost, element count per
// dim), strides_bytes[i] = byte stride of dim i+1.  Box = box[0..rank-1]
// elements.  swizzle_bytes: 128, 64, 32 or 0.  Returns false when the
// encoding is refused (alignment, sizes) or the entry point is missing.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes);

}  // namespace mla
