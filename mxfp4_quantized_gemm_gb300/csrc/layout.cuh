// Device-side offsets of the TILED layout (see include/mxfp4.h).
#pragma once

#include <cstdint>

namespace mx {

// Byte offset of code byte j (0 <= j < Kp/2) of row r in the codes region.
__device__ __forceinline__ size_t tiled_code_offset(int r, int j, int KT) {
  const int rt = r >> 7, i = r & 127, kt = j >> 7, jj = j & 127;
  return (static_cast<size_t>(rt * KT + kt) << 14) + (i << 7) + ((((jj >> 4) ^ (i & 7))) << 4) + (jj & 15);
}
// Byte offset of the scale of row r, block b (0 <= b < Kp/32) in the scales region.
__device__ __forceinline__ size_t tiled_scale_offset(int r, int b, int KT) {
  const int rt = r >> 7, i = r & 127;
  return (static_cast<size_t>(rt * 2 * KT + (b >> 2)) << 9) + ((i & 31) << 4) + ((i >> 5) << 2) + (b & 3);
}

}  // namespace mx
