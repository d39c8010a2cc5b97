// Stores of quantized activations: one lane's chunk of 8 elements (4 code
// bytes) and, from the first lane of each 4-lane group, the group's scale
// byte, in the three activation layouts.  Shared by the standalone quantizer
// and the fused RMSNorm producer.
#pragma once

#include <cstdint>

#include "internal.h"
#include "layout.cuh"

namespace mx {

// Row r, chunk c = elements 8c..8c+7 = code bytes 4c..4c+3, scale block c/4.
// `lead`: this lane stores the block's scale.  kTiled / kBlocked write every
// row and chunk they are called for (padding: zero codes, scale 0x7F);
// kRowMajor writes only rows r < M and bytes inside the row.
template <ActLayout kLayout>
__device__ __forceinline__ void store_act8(uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int r, int M,
                                           int K, int KT, int block_rows, int c, bool lead, uint32_t packed,
                                           uint32_t sbyte) {
  const int nb = (K + 31) >> 5;
  const int blk = c >> 2;
  const bool blk_real = r < M && blk < nb;
  const int j0 = c * 4;
  const uint8_t s = blk_real ? static_cast<uint8_t>(sbyte) : static_cast<uint8_t>(0x7F);
  if (kLayout == ActLayout::kTiled) {
    *reinterpret_cast<uint32_t*>(codes + tiled_code_offset(r, j0, KT)) = packed;
    if (lead) scales[tiled_scale_offset(r, blk, KT)] = s;
  } else if (kLayout == ActLayout::kBlocked) {
    *reinterpret_cast<uint32_t*>(codes + blocked_code_offset(r, j0, KT, block_rows)) = packed;
    if (lead) codes[blocked_scale_offset(r, blk, KT, block_rows)] = s;
  } else if (r < M) {
    const int row_bytes = K >> 1;
    uint8_t* dst = codes + static_cast<size_t>(r) * row_bytes + j0;
    if (j0 + 4 <= row_bytes && (reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (j0 + b < row_bytes) dst[b] = static_cast<uint8_t>(packed >> (8 * b));
    }
    if (lead && blk_real) scales[static_cast<size_t>(r) * nb + blk] = static_cast<uint8_t>(sbyte);
  }
}

}  // namespace mx
