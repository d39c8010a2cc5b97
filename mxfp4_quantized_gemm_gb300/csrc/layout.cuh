// Device-side offsets of the TILED activation layout and of the packed
// weight layout (see include/mxfp4.h).
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

// Activations the library quantizes into its own workspace ("blocked"):
// per (128-row tile mt, k-tile kt) one block of rows * 128 + 1024 bytes at
// (mt * KT + kt) * (rows * 128 + 1024), holding the first `rows` rows of the
// code tile (same swizzle as TILED) followed by the tile's two scale atoms
// (same atom layout; the atoms always take 1024 bytes).  One bulk copy then
// brings a stage its activation codes and scales.  Requires r % 128 < rows.
__device__ __forceinline__ size_t blocked_code_offset(int r, int j, int KT, int rows) {
  const int mt = r >> 7, i = r & 127, kt = j >> 7, jj = j & 127;
  return static_cast<size_t>(mt * KT + kt) * (rows * 128 + 1024) + (i << 7) + (((jj >> 4) ^ (i & 7)) << 4) +
         (jj & 15);
}
__device__ __forceinline__ size_t blocked_scale_offset(int r, int b, int KT, int rows) {
  const int mt = r >> 7, i = r & 127, kt = b >> 3, bb = b & 7;
  return static_cast<size_t>(mt * KT + kt) * (rows * 128 + 1024) + rows * 128 + ((bb >> 2) << 9) +
         ((i & 31) << 4) + ((i >> 5) << 2) + (bb & 3);
}

// Packed weights: blocks of 34816 bytes, one per (256-row pair p, k-tile kt)
// at (p * KT + kt) * 34816, each [code tile of rows 0-127 | code tile of rows
// 128-255 | 2 scale atoms of rows 0-127 | 2 scale atoms of rows 128-255].
// Byte offset of code byte j (0 <= j < Kp/2) of row r:
__device__ __forceinline__ size_t weight_code_offset(int r, int j, int KT) {
  const int p = r >> 8, h = (r >> 7) & 1, i = r & 127, kt = j >> 7, jj = j & 127;
  return static_cast<size_t>(p * KT + kt) * 34816 + (h << 14) + (i << 7) + (((jj >> 4) ^ (i & 7)) << 4) + (jj & 15);
}
// Byte offset of the scale of row r, block b (0 <= b < Kp/32):
__device__ __forceinline__ size_t weight_scale_offset(int r, int b, int KT) {
  const int p = r >> 8, h = (r >> 7) & 1, i = r & 127, kt = b >> 3, bb = b & 7;
  return static_cast<size_t>(p * KT + kt) * 34816 + 32768 + (h << 10) + ((bb >> 2) << 9) + ((i & 31) << 4) +
         ((i >> 5) << 2) + (bb & 3);
}

}  // namespace mx
