// tmap.h -- TMA tensor-map encoding (host).
#pragma once

#include <cstdint>

#include <cuda.h>

#include "lik_internal.h"

namespace lik {

// Encode a tiled tensor map over fp16/bf16/fp32 data of rank 2 or 3 with the
// 128-byte swizzle; dims are innermost first, strides (rank-1 of them) in
// bytes for dims 1.., box in elements.  Out-of-bounds box elements read as
// zero.  Returns false if the driver entry point is unavailable or rejects
// the arguments.
bool encode_tmap_kmajor(CUtensorMap* map, int dtype, const void* base, int rank,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace lik
