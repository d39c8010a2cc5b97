// Fused RMSNorm -> per-1x32 MXFP4 activation producer: the kernel that hands
// the GEMM its input already quantized.  The pages' layer code accepts such a
// (codes, scales) tuple and names a fused RMSNorm as one source of it (sglang
// PR #39598 blog analysis, section 2, apply_weights).  The pages do not print the normalization; it is
// RMSNorm as Zhang and Sennrich (2019) define it, eps inside the root:
//   h = x, or bf16(x + residual) (then also stored as the new residual),
//   y = bf16(h / sqrt(mean(h^2) + eps) * gamma),
// and y is quantized by the same per-block rule as the standalone quantizer
// (quant_math.cuh), so the producer equals RMSNorm-to-bf16 followed by
// mxfp4_quant_act.
//
// One CTA per row (grid-stride over rows); four consecutive lanes hold one
// 32-element scale block.  Pass 1 takes the row (with the residual: adds,
// rounds, stores the sum) and sums squares; one block reduction gives 1/rms;
// pass 2 multiplies by gamma and 1/rms, rounds to bf16 and quantizes.
//   rmsnorm_quant_tma_kernel (K <= 8192, K % 8 == 0, 16-byte aligned rows):
//     thread 0 keeps the CTA's next row in flight as 1-D bulk copies into a
//     2-stage shared-memory ring (x row, then the residual row), refilling a
//     stage right after the row's reduction barrier, so loads overlap the
//     quantization of the row before.  The CTA is sized to the row: each
//     thread owns 2 (up to 256 rows: shorter rows of work) or 4 (more rows:
//     per-row work spread over more elements) 8-element chunks.
//   rmsnorm_quant_kernel<kRegs = true> (other rows with K <= 8192): 256
//     threads, plain vector loads into registers; x is read from HBM once.
//   rmsnorm_quant_kernel<kRegs = false> (K > 8192): pass 2 reads the row
//     again, from L2.
// The element arithmetic uses the Blackwell mixed-precision FMA (bf16 x bf16
// -> f32): squares and h * gamma are exact products.  Squares and sums are
// fp32: rows whose mean square leaves the fp32 range (RMS beyond about 2^63
// or below about 2^-63) are outside the supported range.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "act_store.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "norm_quant.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {

constexpr int kNormThreads = 256;
constexpr int kNormGroup = 4;                                   // chunks a thread loads together
constexpr int kNormRegK = kNormGroup * kNormThreads * 8;        // 8192: rows kept in registers

struct NormArgs {
  const uint16_t* x;
  uint16_t* res;
  const uint16_t* gamma;
  uint16_t* y;
  uint8_t* codes;
  uint8_t* scales;
  int ldx, ldr, ldy;
  float eps;
  int M, K, rows, chunks, KT;
  bool vec_x, vec_r, vec_y, vec_g;
  long long wait_cycles;   // bound of the waits on the row copies (kWaitCycles unless a test lowers it)
};

// bf16(a + b) for 8 values: the packed bf16 add rounds the exact sum once.
__device__ __forceinline__ uint4 add8(uint4 a, uint4 b) {
  uint4 d;
  asm("add.rn.bf16x2 %0, %4, %8;\n\t"
      "add.rn.bf16x2 %1, %5, %9;\n\t"
      "add.rn.bf16x2 %2, %6, %10;\n\t"
      "add.rn.bf16x2 %3, %7, %11;"
      : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
  return d;
}

// acc + the squares of 8 bf16 values, in element order: the mixed-precision
// bf16 x bf16 -> f32 FMA squares exactly and rounds each addition once.
__device__ __forceinline__ float sumsq8(uint4 v, float acc) {
  asm("{\n\t.reg .b16 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      "mov.b32 {l0, h0}, %1;\n\t"
      "mov.b32 {l1, h1}, %2;\n\t"
      "mov.b32 {l2, h2}, %3;\n\t"
      "mov.b32 {l3, h3}, %4;\n\t"
      "fma.rn.f32.bf16 %0, l0, l0, %0;\n\t"
      "fma.rn.f32.bf16 %0, h0, h0, %0;\n\t"
      "fma.rn.f32.bf16 %0, l1, l1, %0;\n\t"
      "fma.rn.f32.bf16 %0, h1, h1, %0;\n\t"
      "fma.rn.f32.bf16 %0, l2, l2, %0;\n\t"
      "fma.rn.f32.bf16 %0, h2, h2, %0;\n\t"
      "fma.rn.f32.bf16 %0, l3, l3, %0;\n\t"
      "fma.rn.f32.bf16 %0, h3, h3, %0;\n\t}"
      : "+f"(acc)
      : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
  return acc;
}

// y = bf16((h * gamma) * rinv) for 8 values: h * gamma is exact in fp32 (a
// product of two bf16 values; adding -0 keeps its sign), so y is rounded once
// to fp32 and once to bf16.  The rinv products go two at a time.
__device__ __forceinline__ void scale_pair(uint32_t h, uint32_t g, uint64_t rr, uint32_t& y) {
  asm("{\n\t.reg .b16 hl, hh, gl, gh;\n\t.reg .f32 pl, ph;\n\t.reg .b64 q;\n\t"
      "mov.b32 {hl, hh}, %1;\n\t"
      "mov.b32 {gl, gh}, %2;\n\t"
      "fma.rn.f32.bf16 pl, hl, gl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 ph, hh, gh, 0f80000000;\n\t"
      "mov.b64 q, {pl, ph};\n\t"
      "mul.rn.f32x2 q, q, %3;\n\t"
      "mov.b64 {pl, ph}, q;\n\t"
      "cvt.rn.bf16x2.f32 %0, ph, pl;\n\t}"
      : "=r"(y)
      : "r"(h), "r"(g), "l"(rr));
}
__device__ __forceinline__ uint4 scale8(uint4 h, uint4 g, float rinv) {
  const uint64_t rr = (static_cast<uint64_t>(__float_as_uint(rinv)) << 32) | __float_as_uint(rinv);
  uint4 y;
  scale_pair(h.x, g.x, rr, y.x);
  scale_pair(h.y, g.y, rr, y.y);
  scale_pair(h.z, g.z, rr, y.z);
  scale_pair(h.w, g.w, rr, y.w);
  return y;
}

// Elements [e0, e0 + 8) of a bf16 row, those below K.
__device__ __forceinline__ void store8(uint16_t* row, int e0, int K, bool vec, uint4 v) {
  if (vec && e0 + 8 <= K) {
    *reinterpret_cast<uint4*>(row + e0) = v;
    return;
  }
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (e0 + i < K) row[e0 + i] = static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1)));
}

// Pass 1 for the chunks c0 + 256 i (i < kNormGroup) of row r: h = x, or
// bf16(x + residual) stored back to the residual; their squares added to ss.
// All loads go out before the first store.
__device__ __forceinline__ void load_group(const NormArgs& a, int r, int c0, uint4 (&h)[kNormGroup], float& ss) {
  const int kc = (a.K + 7) >> 3;
  uint4 q[kNormGroup];
#pragma unroll
  for (int i = 0; i < kNormGroup; ++i) {
    const int c = c0 + i * kNormThreads;
    const bool in = c < kc;
    h[i] = load8_words(a.x, in ? r : a.M, a.M, a.K, a.ldx, c * 8, a.vec_x);
    q[i] = a.res != nullptr ? load8_words(a.res, in ? r : a.M, a.M, a.K, a.ldr, c * 8, a.vec_r)
                            : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kNormGroup; ++i) {
    const int c = c0 + i * kNormThreads;
    if (a.res != nullptr) {
      h[i] = add8(h[i], q[i]);
      if (c < kc) store8(a.res + static_cast<size_t>(r) * a.ldr, c * 8, a.K, a.vec_r, h[i]);
    }
    ss = sumsq8(h[i], ss);
  }
}

// Pass 2 for the chunks c0 + 256 i of row r holding h: y, its optional bf16
// store, quantization and the code / scale stores.  Called by whole warps.
template <bool kTiled>
__device__ __forceinline__ void emit_group(const NormArgs& a, int r, bool real, int c0, const uint4 (&h)[kNormGroup],
                                           const uint4 (&g)[kNormGroup], float rinv) {
  const int kc = (a.K + 7) >> 3;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kNormGroup; ++i) {
    const int c = c0 + i * kNormThreads;
    if (c - lane >= a.chunks) break;    // warp-uniform: the warp's first chunk
    const uint4 yv = real ? scale8(h[i], g[i], rinv) : make_uint4(0, 0, 0, 0);
    if (a.y != nullptr && real && c < kc) store8(a.y + static_cast<size_t>(r) * a.ldy, c * 8, a.K, a.vec_y, yv);
    uint32_t sbyte;
    const uint32_t packed = quantize8_words(yv, sbyte);
    if (c < a.chunks)
      store_act8<kTiled ? ActLayout::kTiled : ActLayout::kRowMajor>(a.codes, a.scales, r, a.M, a.K, a.KT, 0, c,
                                                                     (lane & 3) == 0, packed, sbyte);
  }
}

__device__ __forceinline__ void load_gamma(const NormArgs& a, int c0, uint4 (&g)[kNormGroup]) {
#pragma unroll
  for (int i = 0; i < kNormGroup; ++i) g[i] = load8_words(a.gamma, 0, 1, a.K, 0, (c0 + i * kNormThreads) * 8, a.vec_g);
}

// kRegs: K <= kNormRegK, one group per thread held across both passes.
template <bool kRegs, bool kTiled>
__global__ void __launch_bounds__(kNormThreads, 4) rmsnorm_quant_kernel(NormArgs a) {
  __shared__ float part[2][kNormThreads / 32];
  // kRegs: this thread's gamma chunks, loaded once, read back for every row
  // (only by the thread that wrote them).
  __shared__ uint4 gamma_s[kRegs ? kNormGroup : 1][kNormThreads];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kc = (a.K + 7) >> 3;
  // A programmatic dependent: let the GEMM behind start its set-up now; read
  // x / the residual only once the kernel before this one has completed.
  griddep_launch_dependents();
  griddep_wait();

  uint4 g[kNormGroup];
  if (kRegs) {
    load_gamma(a, tid, g);
#pragma unroll
    for (int i = 0; i < kNormGroup; ++i) gamma_s[kRegs ? i : 0][tid] = g[i];
  }
  int parity = 0;
  for (int r = blockIdx.x; r < a.rows; r += gridDim.x, parity ^= 1) {
    const bool real = r < a.M;    // block-uniform
    float ss = 0.f;
    uint4 h[kNormGroup];
    if (kRegs) {
      if (real) {
        load_group(a, r, tid, h, ss);
      } else {
#pragma unroll
        for (int i = 0; i < kNormGroup; ++i) h[i] = make_uint4(0, 0, 0, 0);
      }
    } else if (real) {
      for (int c0 = tid; c0 - tid < kc; c0 += kNormGroup * kNormThreads) load_group(a, r, c0, h, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) part[parity][warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += part[parity][w];
    const float rinv = rsqrtf(tot / static_cast<float>(a.K) + a.eps);

    if (kRegs) {
#pragma unroll
      for (int i = 0; i < kNormGroup; ++i) g[i] = gamma_s[kRegs ? i : 0][tid];
      emit_group<kTiled>(a, r, real, tid, h, g, rinv);
    } else {
      const uint16_t* src = a.res != nullptr ? a.res : a.x;
      const int ld = a.res != nullptr ? a.ldr : a.ldx;
      const bool vec = a.res != nullptr ? a.vec_r : a.vec_x;
      for (int c0 = tid; c0 - tid < a.chunks; c0 += kNormGroup * kNormThreads) {
#pragma unroll
        for (int i = 0; i < kNormGroup; ++i) {
          const int c = c0 + i * kNormThreads;
          // same thread as the pass-1 store of this chunk: L2 loads see it
          h[i] = load8_words(src, real && c < kc ? r : a.M, a.M, a.K, ld, c * 8, vec);
        }
        load_gamma(a, c0, g);
        emit_group<kTiled>(a, r, real, c0, h, g, rinv);
      }
    }
  }
}

// The bulk-copy variant sizes its CTA to the row: blockDim.x = 32 * W
// threads with W = ceil(chunks / (32 G)), each thread owning the G chunks
// c = tid + blockDim.x * i, i < G -- k-tile warp + W i, code bytes
// 4 * lane .. 4 * lane + 3 of that tile's 128.  G = 4 (at most 8 warps for
// K <= 8192) spreads the per-row work (reduction, 1/rms, offsets) thin for
// many rows; G = 2 (at most 16 warps) shortens each row for a few rows.
constexpr int kTmaMaxWarps = 16;

// Pass 2 of the bulk-copy variant for row r: y, its optional store,
// quantization and the code / scale stores, with the TILED offsets split into
// a per-row part and a per-chunk constant.
template <bool kTiled, bool kY, int kTmaChunks>
__device__ __forceinline__ void emit_row(const NormArgs& a, int r, bool real, const uint4 (&h)[kTmaChunks],
                                         const uint4 (&g)[kTmaChunks], float rinv) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, W = blockDim.x >> 5;
  const int kc = a.K >> 3;
  size_t code_row = 0, scale_row = 0;
  if (kTiled) {
    const int rt = r >> 7, i = r & 127;
    code_row = (static_cast<size_t>(rt) * a.KT << 14) + (i << 7) + (((lane >> 2) ^ (i & 7)) << 4) + ((lane & 3) << 2);
    scale_row = (static_cast<size_t>(rt) * 2 * a.KT << 9) + ((i & 31) << 4) + ((i >> 5) << 2) + ((lane >> 2) & 3);
  }
#pragma unroll
  for (int i = 0; i < kTmaChunks; ++i) {
    const int c = tid + i * static_cast<int>(blockDim.x);
    const int kt = warp + W * i;
    if (kTiled ? kt >= a.KT : c - lane >= a.chunks) break;    // warp-uniform
    const uint4 yv = real ? scale8(h[i], g[i], rinv) : make_uint4(0, 0, 0, 0);
    if (kY && real && c < kc) store8(a.y + static_cast<size_t>(r) * a.ldy, c * 8, a.K, a.vec_y, yv);
    uint32_t sbyte;
    const uint32_t packed = quantize8_words(yv, sbyte);
    if (kTiled) {
      *reinterpret_cast<uint32_t*>(a.codes + code_row + (static_cast<size_t>(kt) << 14)) = packed;
      if ((lane & 3) == 0)
        a.scales[scale_row + (static_cast<size_t>(2 * warp + (lane >> 4) + 2 * W * i) << 9)] =
            real && c < kc ? static_cast<uint8_t>(sbyte) : static_cast<uint8_t>(0x7F);
    } else if (c < a.chunks) {
      store_act8<ActLayout::kRowMajor>(a.codes, a.scales, r, a.M, a.K, a.KT, 0, c, (lane & 3) == 0, packed, sbyte);
    }
  }
}

constexpr int kNormStages = 2;
static __device__ uint32_t g_norm_error;

// Bulk-copy variant: requires K <= kNormRegK, K % 8 == 0 and 16-byte aligned
// x (and residual) rows.  Dynamic shared memory: the ring (kNormStages stages
// of stage_bytes = K * 2, times 2 with a residual), then this CTA's gamma
// chunks (blockDim.x * kTmaChunks * 16 bytes).
template <bool kTiled, bool kRes, bool kY, int kTmaChunks>
__global__ void __launch_bounds__(1024 / kTmaChunks, kTmaChunks) rmsnorm_quant_tma_kernel(NormArgs a, uint32_t stage_bytes) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kNormStages];
  __shared__ __align__(16) float part[2][kTmaMaxWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = static_cast<int>(blockDim.x);
  const int kc = a.K >> 3;
  const uint32_t row_bytes = static_cast<uint32_t>(a.K) * 2;
  uint4* gamma_s = reinterpret_cast<uint4*>(ring + static_cast<size_t>(kNormStages) * stage_bytes);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kNormStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  if (tid < 2 * kTmaMaxWarps) part[tid / kTmaMaxWarps][tid % kTmaMaxWarps] = 0.f;   // slots of absent warps stay 0
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();
  // gamma chunks, each read back only by the thread that stored it
#pragma unroll
  for (int i = 0; i < kTmaChunks; ++i)
    gamma_s[i * T + tid] = load8_words(a.gamma, 0, 1, a.K, 0, (tid + i * T) * 8, a.vec_g);

  // thread 0 keeps the ring full: the row of iteration j (row blockIdx.x +
  // j * gridDim.x) goes to stage j % kNormStages, issued at the start for
  // j < kNormStages, else right after iteration j - kNormStages's barrier.
  auto issue = [&](int r, int s) {
    uint8_t* dst = ring + static_cast<size_t>(s) * stage_bytes;
    mbar_arrive_expect_tx(&full[s], stage_bytes);
    bulk_g2s(dst, a.x + static_cast<size_t>(r) * a.ldx, row_bytes, &full[s]);
    if (kRes) bulk_g2s(dst + row_bytes, a.res + static_cast<size_t>(r) * a.ldr, row_bytes, &full[s]);
  };
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kNormStages; ++s) {
      const int r = blockIdx.x + s * gridDim.x;
      if (r < a.M) issue(r, s);
    }
  }
  const float inv_k = 1.0f / static_cast<float>(a.K);

  bool abort = false;
  int it = 0;
  for (int r = blockIdx.x; r < a.rows; r += gridDim.x, ++it) {
    const bool real = r < a.M;    // real rows are a prefix of this CTA's rows
    const int s = it % kNormStages;
    float ss = 0.f;
    uint4 h[kTmaChunks];
#pragma unroll
    for (int i = 0; i < kTmaChunks; ++i) h[i] = make_uint4(0, 0, 0, 0);
    const uint32_t par = static_cast<uint32_t>(it / kNormStages) & 1u;
    if (real && (a.wait_cycles < kWaitCycles ? mbar_wait_polling(&full[s], par, abort, a.wait_cycles)
                                             : mbar_wait(&full[s], par, abort))) {
      const uint8_t* xs = ring + static_cast<size_t>(s) * stage_bytes;
#pragma unroll
      for (int i = 0; i < kTmaChunks; ++i) {
        const int c = tid + i * T;
        if (c < kc) {
          h[i] = *reinterpret_cast<const uint4*>(xs + c * 16);
          if (kRes) {
            h[i] = add8(h[i], *reinterpret_cast<const uint4*>(xs + row_bytes + c * 16));
            *reinterpret_cast<uint4*>(a.res + static_cast<size_t>(r) * a.ldr + c * 8) = h[i];
          }
          ss = sumsq8(h[i], ss);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) part[it & 1][warp] = ss;
    // every thread is done reading stage s; a timed-out wait anywhere stops the CTA
    if (__syncthreads_or(abort ? 1 : 0)) {
      abort = true;
      break;
    }
    if (tid == 0 && real) {
      const int rn = r + kNormStages * gridDim.x;
      if (rn < a.M) issue(rn, s);
    }
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kTmaMaxWarps; w += 4) {
      const float4 q = *reinterpret_cast<const float4*>(&part[it & 1][w]);
      tot += q.x;
      tot += q.y;
      tot += q.z;
      tot += q.w;
    }
    const float rinv = rsqrtf(tot * inv_k + a.eps);
    uint4 g[kTmaChunks];
#pragma unroll
    for (int i = 0; i < kTmaChunks; ++i) g[i] = gamma_s[i * T + tid];
    emit_row<kTiled, kY, kTmaChunks>(a, r, real, h, g, rinv);
  }
  if (abort && tid == 0) {
    atomicOr(&g_norm_error, kErrTimeout);
    // let the copies still in flight (iterations it .. it + kNormStages - 1,
    // all issued) land before the CTA's memory is reused; these waits take
    // the full bound whatever a.wait_cycles is
    for (int j = it; j < it + kNormStages; ++j) {
      bool again = false;
      if (blockIdx.x + j * gridDim.x < static_cast<unsigned>(a.M))
        mbar_wait(&full[j % kNormStages], static_cast<uint32_t>(j / kNormStages) & 1u, again);
    }
  }
}

static std::atomic<bool> g_norm_attr[16][64];
static std::atomic<uint64_t> g_norm_occ[16][64];

template <bool kTiled, bool kRes, bool kY, int kTmaChunks>
static cudaError_t launch_tma(const NormArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  constexpr int kVariant = (kTiled ? 8 : 0) + (kRes ? 4 : 0) + (kY ? 2 : 0) + (kTmaChunks == 4 ? 1 : 0);
  const int W = (a.chunks + 32 * kTmaChunks - 1) / (32 * kTmaChunks);
  const int T = 32 * W;
  const uint32_t stage_bytes = static_cast<uint32_t>(a.K) * 2 * (kRes ? 2 : 1);
  const int dyn = static_cast<int>(stage_bytes) * kNormStages + T * kTmaChunks * 16;
  auto kern = rmsnorm_quant_tma_kernel<kTiled, kRes, kY, kTmaChunks>;
  std::atomic<bool>& set = g_norm_attr[kVariant][dev.device];
  if (!set.load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kNormStages * kNormRegK * 2 * 2 + kNormRegK * 2);
    if (e != cudaSuccess) return e;
    set.store(true, std::memory_order_release);
  }
  // resident CTAs per SM for this block size and ring, cached (T, dyn) -> count
  std::atomic<uint64_t>& occ = g_norm_occ[kVariant][dev.device];
  const uint64_t key = (static_cast<uint64_t>(T) << 40) | (static_cast<uint64_t>(dyn) << 8);
  uint64_t seen = occ.load(std::memory_order_relaxed);
  int per_sm = static_cast<int>(seen & 0xFF);
  if ((seen & ~uint64_t{0xFF}) != key || per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, T, static_cast<size_t>(dyn));
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 255) per_sm = 255;
    occ.store(key | static_cast<uint64_t>(per_sm), std::memory_order_relaxed);
  }
  int grid = dev.sm_count * per_sm;
  if (grid > a.rows) grid = a.rows;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(T), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(dyn);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, stage_bytes);
}

// G = 2 for up to 256 rows (latency), 4 above (throughput).
template <bool kTiled, bool kRes, bool kY>
static cudaError_t launch_tma_g(const NormArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  return a.M <= 256 ? launch_tma<kTiled, kRes, kY, 2>(a, dev, s) : launch_tma<kTiled, kRes, kY, 4>(a, dev, s);
}

template <bool kTiled>
static cudaError_t launch_tma_any(const NormArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  if (a.res != nullptr)
    return a.y != nullptr ? launch_tma_g<kTiled, true, true>(a, dev, s) : launch_tma_g<kTiled, true, false>(a, dev, s);
  return a.y != nullptr ? launch_tma_g<kTiled, false, true>(a, dev, s) : launch_tma_g<kTiled, false, false>(a, dev, s);
}

uint32_t norm_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_norm_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_norm_error, &zero, sizeof(zero));
  return v;
}

// Bound of the producer's waits on its row copies, in SM clock cycles (0:
// the default kWaitCycles); lowered only by a test to make a wait run out.
static std::atomic<long long> g_norm_wait_cycles{0};

void set_norm_wait_cycles(long long cycles) { g_norm_wait_cycles.store(cycles, std::memory_order_relaxed); }

cudaError_t launch_rmsnorm_quant(const NormQuantProblem& p, const DeviceInfo& dev, cudaStream_t s) {
  NormArgs a{};
  const long long wc = g_norm_wait_cycles.load(std::memory_order_relaxed);
  a.wait_cycles = wc > 0 ? wc : kWaitCycles;
  a.x = static_cast<const uint16_t*>(p.x);
  a.res = static_cast<uint16_t*>(p.residual);
  a.gamma = static_cast<const uint16_t*>(p.gamma);
  a.y = static_cast<uint16_t*>(p.y);
  a.codes = p.codes;
  a.scales = p.scales;
  a.ldx = p.ldx;
  a.ldr = p.ldr;
  a.ldy = p.ldy;
  a.eps = p.eps;
  a.M = p.M;
  a.K = p.K;
  a.KT = static_cast<int>(padded_k(p.K) / kKTile);
  a.rows = p.tiled ? static_cast<int>(padded_rows(p.M)) : p.M;
  a.chunks = p.tiled ? a.KT * (kKTile / 8) : (p.K + 7) / 8;
  auto vec = [](const void* ptr, int ld) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0 && (ld % 8) == 0; };
  a.vec_x = vec(p.x, p.ldx);
  a.vec_r = p.residual != nullptr && vec(p.residual, p.ldr);
  a.vec_y = p.y != nullptr && vec(p.y, p.ldy);
  a.vec_g = vec(p.gamma, 0);
  const bool regs = padded_k(p.K) <= kNormRegK;
  if (regs && (p.K % 8) == 0 && a.vec_x && (p.residual == nullptr || a.vec_r))
    return p.tiled ? launch_tma_any<true>(a, dev, s) : launch_tma_any<false>(a, dev, s);
  int grid = dev.sm_count * 4;
  if (grid > a.rows) grid = a.rows;
  if (p.tiled)
    return regs ? launch_pdl(rmsnorm_quant_kernel<true, true>, grid, kNormThreads, 0, s, a)
                : launch_pdl(rmsnorm_quant_kernel<false, true>, grid, kNormThreads, 0, s, a);
  return regs ? launch_pdl(rmsnorm_quant_kernel<true, false>, grid, kNormThreads, 0, s, a)
              : launch_pdl(rmsnorm_quant_kernel<false, false>, grid, kNormThreads, 0, s, a);
}

}  // namespace mx
