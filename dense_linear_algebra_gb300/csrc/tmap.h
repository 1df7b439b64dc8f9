// tmap.h — 2-D tensor maps of row-major matrices for the tensor copies
// (cp.async.bulk.tensor), encoded by the driver's cuTensorMapEncodeTiled, which is
// fetched once through the runtime (no link against libcuda).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fxtx {

// Map of a matrix of `rows` rows and `cols` elements of `elem` bytes, rows `pitch_bytes`
// apart (a multiple of 16), read in boxes of box_rows x box_bytes (a multiple of 16,
// at most 128 when swizzled). swizzle: 0 (rows land unpermuted), 32, 64 or 128 (the
// swizzle of that width; box_bytes must equal it). Out-of-range elements read as zero.
// False if the driver entry point is missing or refuses the arguments.
bool encode_rows_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t rows, int64_t cols,
                     int64_t pitch_bytes, int elem, int box_rows, int box_bytes, int swizzle);

}  // namespace fxtx
