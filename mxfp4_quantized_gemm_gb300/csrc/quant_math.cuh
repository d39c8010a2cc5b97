// Per-1x32 MXFP4 quantization of bf16 values, the OCP MX conversion the
// pages' per_1x32_f4_quant implements (sglang PR #39598 blog analysis,
// section 2): one E8M0 scale per 32 K-elements with exponent
// floor(log2 amax) - 2, elements rounded to the nearest E2M1 value (ties to
// even) and saturated at +-6.  Shared by the standalone quantizer and the
// GEMM's fused activation quantization.
#pragma once

#include <cstdint>

namespace mx {

// E2M1 magnitude index of a non-negative float by round-to-nearest-even on
// the grid {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating at 6.  Each comparison is
// one midpoint of the grid; a value exactly on a midpoint goes to the
// neighbour with the even code (the comparison is strict towards the odd
// code: 0.25 -> 0, 0.75 -> 2, 1.25 -> 2, 1.75 -> 4, 2.5 -> 4, 3.5 -> 6, 5 -> 6).
__device__ __forceinline__ uint32_t e2m1_magnitude(float a) {
  return static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) +
         static_cast<uint32_t>(a > 1.25f) + static_cast<uint32_t>(a >= 1.75f) +
         static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) + static_cast<uint32_t>(a > 5.0f);
}

// Loads this lane's 8 bf16 values of row r, elements [e0, e0 + 8) (zeros past
// K or for r >= M).
__device__ __forceinline__ void load8_bf16(const uint16_t* __restrict__ x, int r, int M, int K, int ldx, int e0,
                                           bool vec_ok, uint16_t (&v)[8]) {
  if (r < M && vec_ok && e0 + 8 <= K) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(r) * ldx + e0));
    v[0] = q.x & 0xFFFF; v[1] = q.x >> 16; v[2] = q.y & 0xFFFF; v[3] = q.y >> 16;
    v[4] = q.z & 0xFFFF; v[5] = q.z >> 16; v[6] = q.w & 0xFFFF; v[7] = q.w >> 16;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      v[i] = (r < M && e0 + i < K) ? x[static_cast<size_t>(r) * ldx + e0 + i] : static_cast<uint16_t>(0);
  }
}

// Quantizes one 32-element block held by 4 consecutive lanes (8 values each;
// all 32 lanes of the warp call this together).  Returns this lane's 4 code
// bytes (element 2j in the low nibble) and, through sbyte, the block's E8M0
// scale byte (0xFF with zero codes for a block holding Inf or NaN).
__device__ __forceinline__ uint32_t quantize8(const uint16_t (&v)[8], uint32_t& sbyte) {
  // Block amax on the magnitude bits (bf16 magnitudes order like integers;
  // Inf and NaN sort above every finite value).
  uint32_t am = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) am = max(am, static_cast<uint32_t>(v[i] & 0x7FFF));
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
  const uint32_t ef = am >> 7;                 // biased exponent field of amax
  const bool nonfinite = ef == 0xFF;
  // floor(log2 amax) - 2 as an E8M0 byte, clamped at 0 (zero / subnormal amax)
  sbyte = nonfinite ? 0xFFu : (ef > 2 ? ef - 2 : 0u);
  const float inv = __uint_as_float((254u - (nonfinite ? 0u : sbyte)) << 23);   // 2^(127 - sbyte)
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = __uint_as_float(static_cast<uint32_t>(v[i] & 0x7FFF) << 16) * inv;
    uint32_t c = e2m1_magnitude(a) | ((v[i] >> 12) & 8u);
    if (nonfinite) c = 0;
    packed |= c << (4 * i);
  }
  return packed;
}

}  // namespace mx
