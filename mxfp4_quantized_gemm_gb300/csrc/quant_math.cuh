// Per-1x32 MXFP4 quantization of bf16 values, the OCP MX conversion the
// pages' per_1x32_f4_quant implements (sglang PR #39598 blog analysis,
// section 2): one E8M0 scale per 32 K-elements with exponent
// floor(log2 amax) - 2, elements rounded to the nearest E2M1 value (ties to
// even) and saturated at +-6.  Shared by the standalone quantizer, the
// GEMM's fused activation quantization, the fused RMSNorm producer and the
// GEMM's MXFP4 output epilogue.
#pragma once

#include <cstdint>

namespace mx {

// Loads this lane's 8 bf16 values of row r, elements [e0, e0 + 8), as four
// words (element e0 + 2i in the low half of word i; zeros past K or for
// r >= M).  L2-cached loads: x may have been written by the kernel this one
// depends on.
__device__ __forceinline__ uint4 load8_words(const uint16_t* __restrict__ x, int r, int M, int K, int ldx, int e0,
                                             bool vec_ok) {
  if (r >= M) return make_uint4(0, 0, 0, 0);
  const uint16_t* src = x + static_cast<size_t>(r) * ldx + e0;
  if (vec_ok && e0 + 8 <= K) return __ldcg(reinterpret_cast<const uint4*>(src));
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = e0 + 2 * i < K ? src[2 * i] : 0u;
    const uint32_t hi = e0 + 2 * i + 1 < K ? src[2 * i + 1] : 0u;
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The per-block rule, in pieces shared by the 4-lane and the one-thread forms.
//
// amax: bf16 magnitudes order like unsigned integers (Inf and NaN above
// every finite value), so a SIMD max over the sign-cleared halves finds it.
__device__ __forceinline__ uint32_t amax_bits8(uint4 v) {
  const uint32_t m2 = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                               __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m2 & 0xFFFFu, m2 >> 16);
}
// E8M0 byte of a block with bf16 amax bits `am`: floor(log2 amax) - 2,
// clamped at 0 (zero / subnormal amax); 0xFF for a block holding Inf or NaN.
// Also the bf16 bits of the element multiplier 2^(127 - byte).
__device__ __forceinline__ uint32_t block_scale_byte(uint32_t am, uint32_t& inv) {
  const uint32_t ef = am >> 7;                 // biased exponent field of amax
  const bool nonfinite = ef == 0xFF;
  const uint32_t sbyte = nonfinite ? 0xFFu : (ef > 2 ? ef - 2 : 0u);
  inv = (254u - (nonfinite ? 0u : sbyte)) << 7;
  return sbyte;
}
// Codes of 8 bf16 values (element 2j in the low nibble of byte j) times the
// bf16 power of two `inv`: the mixed-precision bf16 x bf16 -> f32 FMA (adding
// -0 keeps the product's sign) gives the exact product (the power is a
// normal number and no flush to zero applies); the hardware E2M1 conversion
// rounds to nearest, ties to even, saturating at 6, and a value that rounds
// to zero keeps its sign (-0 encodes as 0x8).
__device__ __forceinline__ uint32_t e2m1_codes8(uint4 v, uint32_t inv) {
  uint32_t packed;
  // cvt.rn.satfinite.e2m1x2.f32 d, a, b puts a in the high nibble, b in the low.
  asm("{\n\t.reg .b16 s, l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      ".reg .f32 f0, f1, f2, f3, f4, f5, f6, f7;\n\t"
      ".reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.u16.u32 s, %5;\n\t"
      "mov.b32 {l0, h0}, %1;\n\t"
      "mov.b32 {l1, h1}, %2;\n\t"
      "mov.b32 {l2, h2}, %3;\n\t"
      "mov.b32 {l3, h3}, %4;\n\t"
      "fma.rn.f32.bf16 f0, l0, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f1, h0, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f2, l1, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f3, h1, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f4, l2, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f5, h2, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f6, l3, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f7, h3, s, 0f80000000;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, f1, f0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, f3, f2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, f5, f4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, f7, f6;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(packed)
      : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(inv));
  return packed;
}

// Codes of 4 bf16 values (two words) times the bf16 power of two `inv`, as
// e2m1_codes8: 2 bytes, element 2j in the low nibble of byte j.
__device__ __forceinline__ uint32_t e2m1_codes4(uint32_t w0, uint32_t w1, uint32_t inv) {
  uint32_t packed;
  asm("{\n\t.reg .b16 s, l0, h0, l1, h1;\n\t"
      ".reg .f32 f0, f1, f2, f3;\n\t"
      ".reg .b8 b0, b1;\n\t"
      "cvt.u16.u32 s, %3;\n\t"
      "mov.b32 {l0, h0}, %1;\n\t"
      "mov.b32 {l1, h1}, %2;\n\t"
      "fma.rn.f32.bf16 f0, l0, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f1, h0, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f2, l1, s, 0f80000000;\n\t"
      "fma.rn.f32.bf16 f3, h1, s, 0f80000000;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, f1, f0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, f3, f2;\n\t"
      "mov.b32 %0, {b0, b1, 0, 0};\n\t}"
      : "=r"(packed)
      : "r"(w0), "r"(w1), "r"(inv));
  return packed;
}

// Quantizes one 32-element block held by 8 consecutive lanes (4 values each,
// as two bf16 pairs; all 32 lanes of the warp call this together).  Returns
// this lane's 2 code bytes (low 16 bits) and, through sbyte, the block's scale.
__device__ __forceinline__ uint32_t quantize4_words(uint32_t w0, uint32_t w1, uint32_t& sbyte) {
  const uint32_t m2 = __vmaxu2(w0 & 0x7FFF7FFFu, w1 & 0x7FFF7FFFu);
  uint32_t am = max(m2 & 0xFFFFu, m2 >> 16);
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
  uint32_t inv;
  sbyte = block_scale_byte(am, inv);
  const uint32_t packed = e2m1_codes4(w0, w1, inv);
  return sbyte == 0xFFu ? 0u : packed;
}

// Quantizes one 32-element block held by 4 consecutive lanes (8 values each,
// as four bf16 pairs; all 32 lanes of the warp call this together).
// Returns this lane's 4 code bytes and, through sbyte, the block's E8M0
// scale byte (0xFF with zero codes for a block holding Inf or NaN).
__device__ __forceinline__ uint32_t quantize8_words(uint4 v, uint32_t& sbyte) {
  uint32_t am = amax_bits8(v);
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
  am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
  uint32_t inv;
  sbyte = block_scale_byte(am, inv);
  const uint32_t packed = e2m1_codes8(v, inv);   // converted unconditionally, then selected
  return sbyte == 0xFFu ? 0u : packed;
}

// Quantizes one 32-element block held by one thread (32 bf16 values as 16
// pairs, element 2j in the low half of word j): its 16 code bytes and, the
// return value, its scale byte.
__device__ __forceinline__ uint32_t quantize32_words(const uint4 (&v)[4], uint4& codes) {
  const uint32_t am = max(max(amax_bits8(v[0]), amax_bits8(v[1])), max(amax_bits8(v[2]), amax_bits8(v[3])));
  uint32_t inv;
  const uint32_t sbyte = block_scale_byte(am, inv);
  const bool nonfinite = sbyte == 0xFFu;
  codes = make_uint4(nonfinite ? 0u : e2m1_codes8(v[0], inv), nonfinite ? 0u : e2m1_codes8(v[1], inv),
                     nonfinite ? 0u : e2m1_codes8(v[2], inv), nonfinite ? 0u : e2m1_codes8(v[3], inv));
  return sbyte;
}

}  // namespace mx
