// Per-1x32 MXFP4 activation quantization and the one-time repacks.
//
// Quantization follows the OCP MX conversion the pages' per_1x32_f4_quant
// implements (sglang PR #39598 blog analysis, section 2): one E8M0 scale per
// 32 K-elements with exponent floor(log2 amax) - 2, elements rounded to the
// nearest E2M1 value (ties to even) and saturated at +-6.  The repack is the
// Blackwell counterpart of the pages' load-time weight preshuffle and scale
// swizzle (same section: process_weights_after_loading).
#include <cuda_runtime.h>
#include <cstdint>

#include "act_store.cuh"
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {

static __device__ uint32_t g_quant_error;

// A warp owns one 256-element k-tile column kt and the rows r0, r0 + R,
// r0 + 2R, ... of it (R row groups per k-tile: warp gw has kt = gw % KT,
// r0 = gw / KT, the only division); lane l holds elements 8l..8l+7 of the
// k-tile, four lanes form one 32-element block.  Four rows' loads are in
// flight together.  At most 64 registers per thread, so a quantizer block
// fits on an SM next to a resident GEMM CTA.
// kLayout: ActLayout::kRowMajor, kTiled or kBlocked (block_rows rows per
// block; the rows written are 0..rows-1).
template <ActLayout kLayout>
__global__ void __launch_bounds__(256, 4) quant_kernel(const uint16_t* __restrict__ x, int M, int K, int ldx,
                                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                    int rows, int KT, bool vec_ok, int block_rows, int R) {
  const int lane = threadIdx.x & 31;
  const int gw = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  // Launched as a programmatic dependent: let the GEMM behind this kernel
  // start its set-up and weight prefetch now, but touch memory only after the
  // kernel before this one (which may produce x or still read the outputs'
  // buffers) has completed.
  griddep_launch_dependents();
  griddep_wait();
  if (gw >= KT * R) return;   // warp-uniform; the kernel has no block barrier
  const int kt = gw % KT, r0 = gw / KT;
  const int e0 = kt * 256 + lane * 8;
  for (int r = r0; r < rows; r += 4 * R) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int rr = r + j * R;
      v[j] = load8_words(x, rr < rows ? rr : M, M, K, ldx, e0, vec_ok);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int rr = r + j * R;
      if (rr >= rows) break;     // warp-uniform
      uint32_t sbyte;
      const uint32_t packed = quantize8_words(v[j], sbyte);
      store_act8<kLayout>(codes, scales, rr, M, K, KT, block_rows, kt * 32 + lane, (lane & 3) == 0, packed, sbyte);
    }
  }
}

// Repack row-major codes into the TILED codes region: one thread per
// 16-byte output chunk, written in storage order.
__global__ void __launch_bounds__(256) pack_codes_kernel(const uint8_t* __restrict__ codes, int batch, int R,
                                                         int K, uint8_t* __restrict__ packed,
                                                         size_t per_batch, int KT, int64_t chunks_per_batch) {
  const int row_bytes = K >> 1;
  const int64_t total = chunks_per_batch * batch;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(t / chunks_per_batch);
    const int64_t c = t - static_cast<int64_t>(b) * chunks_per_batch;
    const int64_t tile = c >> 10;            // 128 rows x 8 chunks per tile
    const int rem = static_cast<int>(c & 1023);
    const int i = rem >> 3, p = rem & 7;
    const int rt = static_cast<int>(tile / KT), kt = static_cast<int>(tile - static_cast<int64_t>(rt) * KT);
    const int r = rt * 128 + i;
    const int j = kt * 128 + ((p ^ (i & 7)) << 4);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < R && j < row_bytes) {
      const uint8_t* src = codes + (static_cast<size_t>(b) * R + r) * row_bytes + j;
      if (j + 16 <= row_bytes && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        val = __ldg(reinterpret_cast<const uint4*>(src));
      } else {
        uint8_t tmp[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) tmp[q] = (j + q < row_bytes) ? src[q] : static_cast<uint8_t>(0);
        val.x = tmp[0] | (tmp[1] << 8) | (tmp[2] << 16) | (static_cast<uint32_t>(tmp[3]) << 24);
        val.y = tmp[4] | (tmp[5] << 8) | (tmp[6] << 16) | (static_cast<uint32_t>(tmp[7]) << 24);
        val.z = tmp[8] | (tmp[9] << 8) | (tmp[10] << 16) | (static_cast<uint32_t>(tmp[11]) << 24);
        val.w = tmp[12] | (tmp[13] << 8) | (tmp[14] << 16) | (static_cast<uint32_t>(tmp[15]) << 24);
      }
    }
    *reinterpret_cast<uint4*>(packed + static_cast<size_t>(b) * per_batch + static_cast<size_t>(c) * 16) = val;
  }
}

// Repack row-major scales into the TILED scales region: one thread per
// output byte, in storage order; padding gets 0x7F.
__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ scales, int batch, int R,
                                                          int K, uint8_t* __restrict__ packed, size_t per_batch,
                                                          size_t code_bytes, int KT, int64_t bytes_per_batch) {
  const int nb = (K + 31) >> 5;
  const int64_t total = bytes_per_batch * batch;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(t / bytes_per_batch);
    const int64_t o = t - static_cast<int64_t>(b) * bytes_per_batch;
    const int64_t atom = o >> 9;
    const int w = static_cast<int>(o & 511);
    const int i = (w >> 4) + 32 * ((w >> 2) & 3);
    const int rt = static_cast<int>(atom / (2 * KT));
    const int g = static_cast<int>(atom - static_cast<int64_t>(rt) * 2 * KT);
    const int r = rt * 128 + i, blk = g * 4 + (w & 3);
    const uint8_t val = (r < R && blk < nb) ? scales[(static_cast<size_t>(b) * R + r) * nb + blk] : 0x7F;
    packed[static_cast<size_t>(b) * per_batch + code_bytes + static_cast<size_t>(o)] = val;
  }
}

// Repack row-major weight codes and scales into the packed weight blocks:
// one thread per 16-byte output chunk, written in storage order.  A block is
// 2176 chunks: 2048 of codes (two 128-row tiles, 1024 chunks each: row i,
// physical chunk pc holds logical chunk pc ^ (i % 8)), then 128 of scales
// (four 512-byte atoms; byte o of an atom is row (o / 16) + 32 ((o / 4) % 4),
// block o % 4 of its group of four).
__global__ void __launch_bounds__(256) pack_weights_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, int batch, int R,
                                                           int K, uint8_t* __restrict__ packed, int KT,
                                                           int64_t blocks_per_batch) {
  const int row_bytes = K >> 1;
  const int nb = (K + 31) >> 5;
  constexpr int kChunksPerBlock = 2176;
  const int64_t total = static_cast<int64_t>(batch) * blocks_per_batch * kChunksPerBlock;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t blk = t / kChunksPerBlock;
    const int c = static_cast<int>(t - blk * kChunksPerBlock);
    const int bi = static_cast<int>(blk / blocks_per_batch);
    const int64_t pb = blk - static_cast<int64_t>(bi) * blocks_per_batch;
    const int pair = static_cast<int>(pb / KT), kt = static_cast<int>(pb - static_cast<int64_t>(pair) * KT);
    uint8_t v[16];
    if (c < 2048) {
      const int h = c >> 10, rem = c & 1023, i = rem >> 3, pc = rem & 7;
      const int r = pair * 256 + h * 128 + i;
      const int j = kt * 128 + ((pc ^ (i & 7)) << 4);
      const uint8_t* src = codes + (static_cast<size_t>(bi) * R + r) * row_bytes + j;
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = (r < R && j + e < row_bytes) ? src[e] : static_cast<uint8_t>(0);
    } else {
      const int s0 = (c - 2048) * 16;            // byte offset in the 2 KiB scale part
      const int h = s0 >> 10, gq = (s0 >> 9) & 1;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int o = (s0 & 511) + e;
        const int i = (o >> 4) + 32 * ((o >> 2) & 3);
        const int r = pair * 256 + h * 128 + i;
        const int b = kt * 8 + gq * 4 + (o & 3);
        v[e] = (r < R && b < nb) ? scales[(static_cast<size_t>(bi) * R + r) * nb + b] : static_cast<uint8_t>(0x7F);
      }
    }
    uint4 w;
    w.x = v[0] | (v[1] << 8) | (v[2] << 16) | (static_cast<uint32_t>(v[3]) << 24);
    w.y = v[4] | (v[5] << 8) | (v[6] << 16) | (static_cast<uint32_t>(v[7]) << 24);
    w.z = v[8] | (v[9] << 8) | (v[10] << 16) | (static_cast<uint32_t>(v[11]) << 24);
    w.w = v[12] | (v[13] << 8) | (v[14] << 16) | (static_cast<uint32_t>(v[15]) << 24);
    *reinterpret_cast<uint4*>(packed + static_cast<size_t>(blk) * 34816 + static_cast<size_t>(c) * 16) = w;
  }
}

static int grid_for(int64_t work_items, int per_block, const DeviceInfo& dev) {
  int64_t blocks = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

template <typename Kern, typename... Args>
static cudaError_t launch_dependent(Kern k, int grid, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// Warps per k-tile column (R) and blocks for `rows` rows of KT k-tiles.
// Decode-sized inputs (a few rows): at most one 256-thread CTA per SM, which
// fits next to a resident GEMM CTA, so the whole grid starts (and triggers
// its dependent GEMM) at once.  Larger inputs: up to eight CTAs per SM.
static void quant_grid(int rows, int KT, int M, const DeviceInfo& dev, int* R, int* blocks) {
  const int64_t target_warps = static_cast<int64_t>(dev.sm_count) * (M <= kDecodeMaxM ? 1 : 8) * 8;
  int64_t r = target_warps / KT;
  if (r > rows) r = rows;
  if (r < 1) r = 1;
  *R = static_cast<int>(r);
  *blocks = static_cast<int>((static_cast<int64_t>(KT) * r + 7) / 8);
}

cudaError_t launch_quant(const void* x, int M, int K, int ldx, uint8_t* codes, uint8_t* scales, ActLayout layout,
                         int rows_arg, const DeviceInfo& dev, cudaStream_t s) {
  const bool vec_ok = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (ldx % 8) == 0;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  const int KT = static_cast<int>(padded_k(K) / kKTile);
  int R = 1, grid = 1;
  if (layout == ActLayout::kTiled) {
    const int rows = rows_arg > 0 ? rows_arg : static_cast<int>(padded_rows(M));
    quant_grid(rows, KT, M, dev, &R, &grid);
    return launch_dependent(quant_kernel<ActLayout::kTiled>, grid, s, xs, M, K, ldx, codes, scales, rows, KT, vec_ok,
                            0, R);
  }
  if (layout == ActLayout::kBlocked) {
    if (rows_arg <= 0 || rows_arg > kRowTile || (rows_arg < kRowTile && M > rows_arg)) return cudaErrorInvalidValue;
    const int rows = rows_arg == kRowTile ? static_cast<int>(padded_rows(M)) : rows_arg;
    quant_grid(rows, KT, M, dev, &R, &grid);
    return launch_dependent(quant_kernel<ActLayout::kBlocked>, grid, s, xs, M, K, ldx, codes, scales, rows, KT,
                            vec_ok, rows_arg, R);
  }
  const int KTr = static_cast<int>(ceil_div(K, kKTile));
  quant_grid(M, KTr, M, dev, &R, &grid);
  return launch_dependent(quant_kernel<ActLayout::kRowMajor>, grid, s, xs, M, K, ldx, codes, scales, M, KTr, vec_ok,
                          0, R);
}

// Empty kernel launched (normally) after the repack: a programmatic
// dependent launched behind it, such as the GEMM, may prefetch weights before
// its dependency wait, and this guarantees the repack has fully completed.
__global__ void ordering_kernel() {}

cudaError_t launch_ordering(const DeviceInfo& dev, cudaStream_t s) {
  (void)dev;
  ordering_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* codes, const uint8_t* scales, int batch, int R, int K, uint8_t* packed,
                        const DeviceInfo& dev, cudaStream_t s) {
  const int64_t cb = tiled_code_bytes(R, K), sb = tiled_scale_bytes(R, K);
  const size_t per_batch = static_cast<size_t>(cb + sb);
  const int KT = static_cast<int>(padded_k(K) / kKTile);
  const int64_t chunks = cb / 16;
  pack_codes_kernel<<<grid_for(chunks * batch, 256, dev), 256, 0, s>>>(codes, batch, R, K, packed, per_batch, KT,
                                                                       chunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pack_scales_kernel<<<grid_for(sb * batch, 256, dev), 256, 0, s>>>(scales, batch, R, K, packed, per_batch,
                                                                    static_cast<size_t>(cb), KT, sb);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ordering_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t launch_pack_weights(const uint8_t* codes, const uint8_t* scales, int batch, int N, int K,
                                uint8_t* packed, const DeviceInfo& dev, cudaStream_t s) {
  const int KT = static_cast<int>(padded_k(K) / kKTile);
  const int64_t blocks = weight_rows(N) / kPairRows * KT;
  pack_weights_kernel<<<grid_for(blocks * batch * 2176, 256, dev), 256, 0, s>>>(codes, scales, batch, N, K, packed, KT,
                                                                                blocks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ordering_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

uint32_t quant_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(zero));
  return v;
}

}  // namespace mx
