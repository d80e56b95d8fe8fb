// Host access to the driver's tensor-map encoder (cuTensorMapEncodeTiled), fetched once through the
// runtime's driver entry-point query so that the library links against the runtime only.
#pragma once

#include <cuda.h>

namespace ers {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The encoder, or null when the driver offers none (callers then report the path as unsupported).
EncodeTiledFn tma_encode_fn();

}  // namespace ers
