// tmap.h -- TMA tensor maps for the tensor-core kernels.
#pragma once

#include <cuda.h>

namespace spattn {

// [BH][rows * dview][D] bf16 seen as {D, dview, rows, BH}: element (x, r, q, bh) is
// row q * dview + r of head bh.  Boxes of box_rows rows (q) x 64 columns, one residue r,
// 128-byte swizzle, zero fill past `rows`.  dview = 1 is the plain [BH][rows][D].
// Returns false when the driver's encoder is unavailable or rejects the map.
bool make_map(CUtensorMap* map, const void* base, int D, long long rows, long long BH,
              long long dview = 1, int box_rows = 128);

}  // namespace spattn
