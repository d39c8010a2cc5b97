// Pieces shared by the two W4A4 GEMM kernels (gemm.cu: M > 64, decode.cu:
// M <= 64): the shared-memory stage geometry, the stream-K split of the
// (output tile, k-step) iteration space, and the bias + bf16 output stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {

constexpr int kTileN = 256;          // weight rows per output tile (the MMA's N)
constexpr int kThreads = 320;        // producer warp, MMA warp, 8 epilogue warps
constexpr int kEpiThreads = 256;
constexpr int kMaxSmem = 232448;     // 227 KiB of dynamic shared memory per CTA

// One pipeline stage = one 256-wide k-step of one output tile: the packed
// weight block of the tile's 256 rows (two 16 KiB code tiles, then 2 x 2
// scale atoms: one bulk copy), kRowsA activation rows of codes and two
// activation scale atoms.
template <int kRowsA>
struct Cfg {
  static constexpr int kW = kWeightBlockBytes;    // 256 weight rows: codes + scales
  // Only the first kRowsA activation rows are loaded and reserved per stage.
  // The M = 128 MMA reads 16 KiB from the activation offset; for kRowsA <
  // 128 the rows past kRowsA come from whatever follows (the rest of the
  // stage, the next stage, or a tail pad after the last one, so every read
  // stays inside the allocation) and feed only accumulator rows that are
  // never read.
  static constexpr int kALoad = kRowsA * 128;
  static constexpr int kA = kALoad;
  static constexpr int kTailPad = kTileBytes - kALoad;
  static constexpr int kSA = 1024;                // 2 activation scale atoms
  static constexpr int kStageBytes = kW + kA + kSA;
  static constexpr int kStagesFit = (kMaxSmem - 1024 - 512 - kTailPad) / kStageBytes;
  // The decode shapes (kRowsA <= 64) keep four stages: enough to stream the
  // weights at the HBM rate, and at the end of a call the MMAs of the stages
  // still buffered hold the SM (and keep the next call's CTA off it) for
  // less time than with five (measured: 3 stages 2.7% slower on the decode
  // sweep, 5 stages 1% slower).
  static constexpr int kMaxStages = kRowsA <= 64 ? 4 : 8;
  static constexpr int kStages = kStagesFit > kMaxStages ? kMaxStages : kStagesFit;
  static constexpr int kRing = kStages * kStageBytes + kTailPad;
  static constexpr int kSmem = kRing + 1024 + 512;
  // TMEM: the 128 x 256 fp32 accumulator in columns 0..255, then one
  // 32-column scale slot per ring stage (activation scales in its first 8
  // columns, weight scales in the next 16).  A stage's scales never share
  // columns with the stage before it, so copying them in does not wait for
  // the previous stage's MMAs to finish reading theirs.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSfBase = 256, kSfSlot = 32, kSfbOff = 8;
  static_assert(kSfBase + kStages * kSfSlot <= kTmemCols, "scale slots exceed TMEM");
};

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
// v + bias[n], or v itself without a bias (no + 0: a -0 result stays -0, the
// same in every store path).
__device__ __forceinline__ float with_bias(const uint16_t* bias, int n, float v) {
  return bias != nullptr ? v + bf16_bits_to_float(__ldg(bias + n)) : v;
}

// Balanced stream-K split: CTA c owns iterations [sk_begin(c), sk_begin(c+1)).
__device__ __forceinline__ int sk_begin(int c, int total, int grid) {
  return static_cast<int>((static_cast<long long>(c) * total) / grid);
}
// CTA whose range holds iteration `it`.
__device__ __forceinline__ int sk_owner(int it, int total, int grid) {
  int c = static_cast<int>((static_cast<long long>(it) * grid) / total);
  while (c + 1 < grid && sk_begin(c + 1, total, grid) <= it) ++c;
  while (c > 0 && sk_begin(c, total, grid) > it) --c;
  return c;
}

// Where the results go: bf16 [M][ldo]; or (qcodes != null) the MXFP4
// quantization of those bf16 values, row-major codes [M][N/2] and scales
// [M][ceil(N/32)] (N even); or (splitcat set) the split + cat form: the
// columns are H = N / (s1 + s2) groups of s1 + s2, the first s1 of group h
// go to cat[m][h][0, s1) and the other s2 to split[m][h][0, s2), and z[m][h]
// (s3 values) is copied to cat[m][h][s1, s1 + s3).  s1, s2, s3 are
// multiples of 8 and cat, split, z 16-byte aligned.
struct OutView {
  __nv_bfloat16* out;
  const __nv_bfloat16* bias;   // [N] or null
  int ldo, N;
  uint8_t* qcodes;
  uint8_t* qscales;
  __nv_bfloat16* cat;          // [M][H][s1 + s3]
  __nv_bfloat16* split;        // [M][H][s2]
  const __nv_bfloat16* z;      // [M][H][s3]
  int s1, s2, s3;
  int splitcat;
};

// Split + cat form: the bf16 results of row m, columns n .. n + w - 1 (w = 4
// or 8, never crossing a group part since n, s1 and s2 are multiples of 8
// or n % 8 + w <= 8), to their place in cat or split; with them, the z
// values of the same row and group at offsets j, j + G, j + 2G, ... (j the
// columns' offset in the group, G = s1 + s2) are copied into cat, so the
// groups' columns together copy all of z[m][h].
template <int W>
__device__ __forceinline__ void store_sc(const OutView& o, int m, int n, const uint32_t (&w)[W / 2]) {
  const int G = o.s1 + o.s2, H = o.N / G;
  const int h = n / G, j = n - h * G;
  const size_t gi = static_cast<size_t>(m) * H + h;
  __nv_bfloat16* dst = j < o.s1 ? o.cat + gi * (o.s1 + o.s3) + j : o.split + gi * o.s2 + (j - o.s1);
  if constexpr (W == 8)
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  else
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
  for (int jz = j; jz < o.s3; jz += G) {
    const __nv_bfloat16* src = o.z + gi * o.s3 + jz;
    __nv_bfloat16* d2 = o.cat + gi * (o.s1 + o.s3) + o.s1 + jz;
    if constexpr (W == 8)
      *reinterpret_cast<uint4*>(d2) = __ldg(reinterpret_cast<const uint4*>(src));
    else
      *reinterpret_cast<uint2*>(d2) = __ldg(reinterpret_cast<const uint2*>(src));
  }
}

// MXFP4 output: the 32 outputs of row m from column n (a multiple of 32) +
// bias, rounded to bf16 exactly as the bf16 store rounds them, then
// quantized as one 1x32 block (columns past N count as zeros) by the
// thread that holds them.
__device__ __forceinline__ void store_chunk_q(const OutView& o, int m, int n, const float (&v)[32]) {
  if (n >= o.N) return;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(o.bias);
  uint32_t w[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int c = n + 2 * j;
    const float lo = c < o.N ? with_bias(bias, c, v[2 * j]) : 0.f;
    const float hi = c + 1 < o.N ? with_bias(bias, c + 1, v[2 * j + 1]) : 0.f;
    w[j] = pack_bf16x2(lo, hi);
  }
  const uint4 blk[4] = {make_uint4(w[0], w[1], w[2], w[3]), make_uint4(w[4], w[5], w[6], w[7]),
                        make_uint4(w[8], w[9], w[10], w[11]), make_uint4(w[12], w[13], w[14], w[15])};
  uint4 codes;
  const uint32_t sbyte = quantize32_words(blk, codes);
  const int row_bytes = o.N >> 1;
  uint8_t* dst = o.qcodes + static_cast<size_t>(m) * row_bytes + (n >> 1);
  if (n + 32 <= o.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
    *reinterpret_cast<uint4*>(dst) = codes;
  } else {
    const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int b = 0; b < 16; ++b)
      if ((n >> 1) + b < row_bytes) dst[b] = static_cast<uint8_t>(cw[b >> 2] >> (8 * (b & 3)));
  }
  o.qscales[static_cast<size_t>(m) * ((o.N + 31) >> 5) + (n >> 5)] = static_cast<uint8_t>(sbyte);
}

// 32 consecutive outputs of row m starting at column n: + bias, bf16, store.
__device__ __forceinline__ void store_chunk_bf16(const OutView& o, int m, int n, const float (&v)[32]) {
  __nv_bfloat16* dst = o.out + static_cast<size_t>(m) * o.ldo + n;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(o.bias);
  if (n + 32 <= o.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int c = 0; c < 32; c += 8) {
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = with_bias(bias, n + c + i, v[c + i]);
      uint4 w;
      w.x = pack_bf16x2(x[0], x[1]);
      w.y = pack_bf16x2(x[2], x[3]);
      w.z = pack_bf16x2(x[4], x[5]);
      w.w = pack_bf16x2(x[6], x[7]);
      *reinterpret_cast<uint4*>(dst + c) = w;
    }
  } else {
    for (int c = 0; c < 32; ++c)
      if (n + c < o.N) dst[c] = __float2bfloat16_rn(with_bias(bias, n + c, v[c]));
  }
}

// 32 consecutive outputs of row m from column n (a multiple of 8): + bias,
// bf16, to the split + cat outputs, 8 columns at a time.
__device__ __forceinline__ void store_chunk_sc(const OutView& o, int m, int n, const float (&v)[32]) {
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(o.bias);
#pragma unroll
  for (int c = 0; c < 32; c += 8) {
    if (n + c >= o.N) break;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = pack_bf16x2(with_bias(bias, n + c + 2 * i, v[c + 2 * i]), with_bias(bias, n + c + 2 * i + 1, v[c + 2 * i + 1]));
    store_sc<8>(o, m, n + c, w);
  }
}

// The same, or for MXFP4 output (o.qcodes set) its quantization (n is then a
// multiple of 32), or the split + cat form (o.splitcat set).
__device__ __forceinline__ void store_chunk(const OutView& o, int m, int n, const float (&v)[32]) {
  if (o.qcodes != nullptr)
    store_chunk_q(o, m, n, v);
  else if (o.splitcat)
    store_chunk_sc(o, m, n, v);
  else
    store_chunk_bf16(o, m, n, v);
}

// 4 consecutive outputs of row m starting at column n: + bias, bf16, store.
// 4 consecutive outputs of row m from column n (a multiple of 4): + bias,
// bf16, to the split + cat outputs.
__device__ __forceinline__ void store_quad_sc(const OutView& o, int m, int n, float4 v) {
  if (n >= o.N) return;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(o.bias);
  const uint32_t w[2] = {pack_bf16x2(with_bias(bias, n, v.x), with_bias(bias, n + 1, v.y)),
                         pack_bf16x2(with_bias(bias, n + 2, v.z), with_bias(bias, n + 3, v.w))};
  store_sc<4>(o, m, n, w);
}

__device__ __forceinline__ void store_quad(const OutView& o, int m, int n, float4 v) {
  if (n >= o.N) return;
  __nv_bfloat16* dst = o.out + static_cast<size_t>(m) * o.ldo + n;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(o.bias);
  float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (n + i < o.N) x[i] = with_bias(bias, n + i, x[i]);
  if (n + 4 <= o.N && (reinterpret_cast<uintptr_t>(dst) & 7) == 0) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (n + i < o.N) dst[i] = __float2bfloat16_rn(x[i]);
  }
}

__device__ __forceinline__ void store_quad_any(const OutView& o, int m, int n, float4 v) {
  if (o.splitcat)
    store_quad_sc(o, m, n, v);
  else
    store_quad(o, m, n, v);
}

// One stage of the MMA pipeline: the tcgen05.cp copies of its scales into
// TMEM -- activation scales (2 atoms) at column sfa_col, weight scales (2
// atoms x 2 row halves; atom of half q, block group a at q * 1024 + a * 512
// after the codes) at sfb_col -- then the four K = 64 block-scaled MMAs into
// the accumulator [128 act rows x 256 weight rows] at `tmem`; `accumulate` =
// 0 starts a new tile.  The copies write only scale columns, so at a tile
// boundary they may go out before the accumulator is free again.
// `copy_a` = false reuses activation scales already at sfa_col (copied for
// an earlier tile of the same activation rows).
template <typename C>
__device__ __forceinline__ void issue_stage_scales_sfa(uint32_t tmem, uint32_t stage_base, uint32_t sfb_col,
                                                       uint32_t sfa_col, bool copy_a) {
  const uint32_t sfa = tmem + sfa_col;
  const uint32_t sfb = tmem + sfb_col;
  const uint32_t sw_s = stage_base + 2 * kTileBytes, sa_s = stage_base + C::kW + C::kA;
  if (copy_a) {
    tmem_cp_scales(sfa + 0, sdesc_scales(sa_s));
    tmem_cp_scales(sfa + 4, sdesc_scales(sa_s + 512));
  }
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int q = 0; q < 2; ++q) tmem_cp_scales(sfb + a * 8 + q * 4, sdesc_scales(sw_s + q * 1024 + a * 512));
}
template <typename C>
__device__ __forceinline__ void issue_stage_mmas_sfa(uint32_t tmem, uint32_t stage_base, uint32_t sfb_col,
                                                     uint32_t sfa_col, uint32_t accumulate) {
  const uint32_t sfa = tmem + sfa_col;
  const uint32_t sfb = tmem + sfb_col;
  const uint32_t w_s = stage_base, a_s = stage_base + C::kW;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t id = idesc_mxf4(128, kTileN, (q & 1) * 2, (q & 1) * 2);
    mma_mxf4(tmem, sdesc_sw128(a_s + 32 * q), sdesc_sw128(w_s + 32 * q), id, sfa + 4 * (q >> 1), sfb + 8 * (q >> 1),
             (accumulate != 0 || q != 0) ? 1u : 0u);
  }
}

template <typename C>
__device__ __forceinline__ void issue_stage_mma_sfa(uint32_t tmem, uint32_t stage_base, uint32_t sfb_col,
                                                    uint32_t sfa_col, bool copy_a, uint32_t accumulate) {
  issue_stage_scales_sfa<C>(tmem, stage_base, sfb_col, sfa_col, copy_a);
  issue_stage_mmas_sfa<C>(tmem, stage_base, sfb_col, sfa_col, accumulate);
}

// The same with both scale sets in ring slot `slot`'s 32 TMEM columns.
template <typename C>
__device__ __forceinline__ void issue_stage_scales(uint32_t tmem, uint32_t stage_base, int slot) {
  const uint32_t sfa = tmem + C::kSfBase + static_cast<uint32_t>(slot) * C::kSfSlot;
  issue_stage_scales_sfa<C>(tmem, stage_base, sfa + C::kSfbOff - tmem, sfa - tmem, true);
}
template <typename C>
__device__ __forceinline__ void issue_stage_mmas(uint32_t tmem, uint32_t stage_base, int slot, uint32_t accumulate) {
  const uint32_t sfa_col = C::kSfBase + static_cast<uint32_t>(slot) * C::kSfSlot;
  issue_stage_mmas_sfa<C>(tmem, stage_base, sfa_col + C::kSfbOff, sfa_col, accumulate);
}
template <typename C>
__device__ __forceinline__ void issue_stage_mma(uint32_t tmem, uint32_t stage_base, int slot, uint32_t accumulate) {
  issue_stage_scales<C>(tmem, stage_base, slot);
  issue_stage_mmas<C>(tmem, stage_base, slot, accumulate);
}

// Launch as a programmatic dependent of the previous kernel in the stream.
template <typename Kern, typename Args>
static cudaError_t launch_pdl(Kern k, int grid, int threads, int smem, cudaStream_t s, const Args& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

}  // namespace mx
