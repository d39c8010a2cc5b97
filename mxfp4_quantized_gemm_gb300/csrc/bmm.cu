// A16WFP4 batched matmul for the MLA absorbed K-up / V-up projections of
// sglang PR #34317 "[AMD] [GLM5] use tuned MXFP4 kernels for MLA absorbed
// BMM" (Modifications): bf16 activations against FP4 weights with E8M0
// scales, the V-up result written batch-major [M, B, N] directly.
//
//   r[b][m][n] = bf16_RNE( sum_k x[b][m][k] * deq(W_b)[n][k] )
//
// One CTA owns (batch b, a tile of BN weight rows) and loops over the M
// tiles.  Its weight tile is dequantized once into shared memory as bf16 in
// the 128-byte-swizzled K-major operand image (e2m1 * 2^(s-127) is exact in
// bf16 for every scale the format can hold except the extreme subnormals),
// and stays resident; activations stream through a ring of 128 x 64 bf16
// slabs (as deep as the shared memory left over allows) fed by TMA tensor
// loads; one thread issues tcgen05.mma.kind::f16 (bf16 x bf16 -> fp32 TMEM);
// eight warps drain the double-buffered accumulator while the next M tile is
// multiplied, staging each 32-row x 32-column piece in shared memory so that
// every warp store writes whole 64-byte row segments.  For 256 < K <= 512
// (the V-up shape) a second kernel keeps the 128-row weight tile in TMEM as
// the MMA's A operand instead, which leaves shared memory to a deeper x ring
// and lets one commit cover four slabs (see a16wfp4_bmm_ts_kernel).  Both
// kernels are programmatic dependent launches: the weight tile is
// dequantized before the wait for the kernel ahead of it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"

namespace mx {

static __device__ uint32_t g_bmm_error;

constexpr int kBmmThreads = 320;           // producer warp, MMA warp, 8 epilogue warps
constexpr int kBmmMaxStages = 8;
constexpr int kSlabBytes = 128 * 128;      // 128 rows x 64 bf16
constexpr int kPieceCols = 32;             // epilogue piece: 32 rows x 32 columns
constexpr int kStageOutBytes = 32 * kPieceCols * 2;   // per epilogue warp

struct BmmArgs {
  const uint8_t* w_packed;
  __nv_bfloat16* out;
  int B, M, N, K, KS;        // KS = K / 64 slabs
  int BN, n_tiles, m_tiles, m_per_cta;
  int stages;                // x ring depth (stages of G slabs)
  int G;                     // slabs per ring stage (a16wfp4_bmm_ts_kernel; 1 otherwise)
  size_t w_batch_bytes;      // packed weight bytes of one batch
  int KT;                    // Kp / 256 of the packed weights
  bool batch_major;
  bool vec_out;              // out 16-byte aligned and N % 8 == 0: 16-byte output stores
};

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 2^(s-127) as a float for an E8M0 byte (0xFF -> NaN).
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
  if (s == 0xFF) return __uint_as_float(0x7FC00000u);
  if (s == 0) return __uint_as_float(0x00400000u);   // 2^-127, a float subnormal
  return __uint_as_float(s << 23);
}

// The two E2M1 values of a code byte (low nibble first), each times the
// block scale, as a bf16 pair.  The hardware conversion to f16 is exact (every
// E2M1 value is an f16), the product is formed in fp32 and rounded once.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t byte, float sc) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "r"(byte));
  const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFF)));
  const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  return pack_bf16x2(lo * sc, hi * sc);
}

__global__ void __launch_bounds__(kBmmThreads, 1) a16wfp4_bmm_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                    const BmmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = g.BN;
  const int stages = g.stages;
  uint8_t* wsm = smem;                                       // KS slabs of BN rows x 128 B
  uint8_t* xsm = smem + static_cast<size_t>(g.KS) * BN * 128; // ring of x slabs
  uint8_t* osm = xsm + stages * kSlabBytes;                   // 8 x kStageOutBytes output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(osm + 8 * kStageOutBytes);
  uint64_t* empty = full + kBmmMaxStages;
  uint64_t* acc_full = empty + kBmmMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x % g.n_tiles;
  const int b = blockIdx.x / g.n_tiles;
  const int mt0 = blockIdx.y * g.m_per_cta;
  const int mt1 = min(g.m_tiles, mt0 + g.m_per_cta);
  const uint32_t tmem_cols = 2 * BN;
  bool abort = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kBmmThreads - 64);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  // The next kernel in the stream waits for this one to complete before it
  // touches memory, so it may start launching now.
  if (threadIdx.x == 0) griddep_launch_dependents();

  // ---- dequantize this CTA's weight tile into the swizzled bf16 image.  The
  // packed weights are never written by the kernel before this one, so this
  // runs before the dependency wait; four items' loads are in flight per
  // thread.  Item = (weight row, 32-element block): 16 code bytes + 1 scale.
  {
    const uint8_t* wb = g.w_packed + static_cast<size_t>(b) * g.w_batch_bytes;
    const int nblk = g.K >> 5;
    const int items = BN * nblk;
    for (int it0 = threadIdx.x; it0 < items; it0 += 4 * kBmmThreads) {
      uint4 c[4];
      uint32_t sb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int it = it0 + j * kBmmThreads;
        if (it < items) {
          const int nl = it / nblk, blk = it - nl * nblk;
          const int n = nt * BN + nl;
          c[j] = __ldg(reinterpret_cast<const uint4*>(wb + weight_code_offset(n, blk * 16, g.KT)));
          sb[j] = __ldg(wb + weight_scale_offset(n, blk, g.KT));
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int it = it0 + j * kBmmThreads;
        if (it >= items) break;
        const int nl = it / nblk, blk = it - nl * nblk;
        const float sc = e8m0_to_float(sb[j]);
        const uint32_t w32[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
        uint32_t o[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) o[q] = dequant_pair((w32[q >> 2] >> (8 * (q & 3))) & 0xFF, sc);
        // 32 elements = 4 swizzled 16-byte chunks of one slab row
        const int k0 = blk * 32;
        const int slab = k0 >> 6;
        const int chunk0 = (k0 & 63) >> 3;
        uint8_t* row = wsm + static_cast<size_t>(slab) * BN * 128 + nl * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int phys = (chunk0 + cc) ^ (nl & 7);
          *reinterpret_cast<uint4*>(row + phys * 16) =
              make_uint4(o[4 * cc], o[4 * cc + 1], o[4 * cc + 2], o[4 * cc + 3]);
        }
      }
    }
    fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // x and the output may be written / read by the kernel before this one.
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer: x slabs by TMA
      uint32_t ls = 0;
      for (int mt = mt0; mt < mt1; ++mt) {
        for (int ks = 0; ks < g.KS; ++ks, ++ls) {
          const int s = ls % stages;
          const uint32_t ph = (ls / stages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
          mbar_arrive_expect_tx(&full[s], kSlabBytes);
          tma_load_3d(xsm + s * kSlabBytes, &xmap, ks * 64, mt * 128, b, &full[s]);
        }
        if (abort) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer.  Its MMAs are small (128 x BN x 16), so the scalar
      // work between them matters: the ring slot and phase advance by
      // counters, and the shared-memory descriptors by their address field
      // (an operand's address >> 4 sits in the low bits; every operand here
      // lies below 256 KiB, so the sums never carry out of the field).
      const uint32_t idesc = idesc_bf16(128, BN);
      const uint64_t xdesc0 = sdesc_sw128(smem_u32(xsm));
      const uint64_t wdesc0 = sdesc_sw128(smem_u32(wsm));
      constexpr uint64_t kSlabStep = kSlabBytes >> 4, kKStep = 32 >> 4;
      const uint64_t wslab_step = static_cast<uint64_t>(BN) * 128 >> 4;
      int s = 0;
      uint32_t ph = 0;
      int i = 0;
      for (int mt = mt0; mt < mt1 && !abort; ++mt, ++i) {
        const int buf = i & 1;
        const uint32_t use = i >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort)) break;
        tc_fence_after();
        const uint32_t acc = tmem + buf * BN;
        uint64_t wdesc = wdesc0;
        for (int ks = 0; ks < g.KS; ++ks) {
          if (!mbar_wait(&full[s], ph, abort)) break;
          tc_fence_after();
          const uint64_t xdesc = xdesc0 + static_cast<uint64_t>(s) * kSlabStep;
          mma_bf16(acc, xdesc, wdesc, idesc, ks != 0);
#pragma unroll
          for (int j = 1; j < 4; ++j) mma_bf16(acc, xdesc + j * kKStep, wdesc + j * kKStep, idesc, 1u);
          mma_commit(&empty[s]);
          wdesc += wslab_step;
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        mma_commit(&acc_full[buf]);
      }
      // TMEM is freed only after the last drain has read both accumulators.
      for (int k = i - 2 < 0 ? 0 : i - 2; k < i; ++k) mbar_wait(&acc_empty[k & 1], (k >> 1) & 1, abort);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  } else {
    // ---- epilogue: warp w (2..9) drains accumulator rows 32 (w % 4).. and
    // columns [h BN/2, (h+1) BN/2) (h = 0 for warps 2..5, 1 for 6..9) in
    // pieces of 32 columns.  Lane l converts row l's piece to bf16 into the
    // warp's staging area (16-byte chunk c of row r at chunk c ^ ((r / 2) % 4):
    // conflict-free both ways); then each pass stores 8 rows x 64 contiguous
    // bytes.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* stg = osm + (warp - 2) * kStageOutBytes;
    auto row_ptr = [&](int m) -> __nv_bfloat16* {
      return g.batch_major ? g.out + (static_cast<size_t>(m) * g.B + b) * g.N
                           : g.out + (static_cast<size_t>(b) * g.M + m) * g.N;
    };
    const int half = BN >> 1;
    int i = 0;
    for (int mt = mt0; mt < mt1; ++mt, ++i) {
      const int buf = i & 1;
      const uint32_t use = i >> 1;
      const bool ok = mbar_wait(&acc_full[buf], use & 1, abort);
      tc_fence_after();
      const int mrow0 = mt * 128 + q * 32;
      for (int c0 = h * half; c0 < (h + 1) * half; c0 += kPieceCols) {
        uint32_t r[32];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c0,
                  *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c0 + 16,
                  *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
        tmem_wait_ld();
        if (c0 + kPieceCols >= (h + 1) * half) {
          tc_fence_before();
          mbar_arrive(&acc_empty[buf]);          // this warp's share of the accumulator is read
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint4 w;
          w.x = ok ? pack_bf16x2(__uint_as_float(r[8 * ch]), __uint_as_float(r[8 * ch + 1])) : 0u;
          w.y = ok ? pack_bf16x2(__uint_as_float(r[8 * ch + 2]), __uint_as_float(r[8 * ch + 3])) : 0u;
          w.z = ok ? pack_bf16x2(__uint_as_float(r[8 * ch + 4]), __uint_as_float(r[8 * ch + 5])) : 0u;
          w.w = ok ? pack_bf16x2(__uint_as_float(r[8 * ch + 6]), __uint_as_float(r[8 * ch + 7])) : 0u;
          *reinterpret_cast<uint4*>(stg + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4)) = w;
        }
        __syncwarp();
#pragma unroll
        for (int pss = 0; pss < 4; ++pss) {
          const int rr = pss * 8 + (lane >> 2), ch = lane & 3;
          const int m = mrow0 + rr;
          const int n = nt * BN + c0 + ch * 8;
          const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * 64 + ((ch ^ ((rr >> 1) & 3)) << 4));
          if (m < g.M && n < g.N) {
            __nv_bfloat16* dst = row_ptr(m) + n;
            if (g.vec_out && n + 8 <= g.N) {
              *reinterpret_cast<uint4*>(dst) = w;
            } else {
              const uint32_t hw[4] = {w.x, w.y, w.z, w.w};
              for (int e = 0; e < 8 && n + e < g.N; ++e)
                reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(hw[e >> 1] >> (16 * (e & 1)));
            }
          }
        }
        __syncwarp();
      }
    }
  }
  if (abort) atomicOr(&g_bmm_error, kErrTimeout);
}

// ------------------------------------------------- weights resident in TMEM
// For 256 < K <= 512, where a bf16 image of 256 weight rows would not fit in
// shared memory next to an x ring, and one of 128 rows would leave a ring of
// only five slabs: the CTA's 128 weight rows, dequantized to bf16, stay in
// TMEM as the MMA's A operand (columns 256 .. 256 + K/2, two bf16 per
// column), so shared memory holds only the x ring (twelve slabs, in stages
// of up to four) and the epilogue staging.  The small MMAs need the stages:
// committing after every four 128 x 128 x 16 MMAs holds the tensor pipe to
// about one commit group per 255 ns, while sixteen per commit run at 37 ns
// each (the V-up call at B = 64, M = 4096 takes 71 us instead of 91 with one
// slab per stage).  The MMA forms the transposed tile
//   D[n][m] = sum_k W[n][k] x[m][k]
// with the 128 weight rows in lanes and 128 activation rows in columns,
// double-buffered in columns 0..255; the epilogue transposes each 32 x 32
// piece (lane pairs exchange values with one shuffle per two columns, then
// the words go through the warp's staging area) so that every store still
// writes 64 contiguous bytes of an output row.
constexpr int kTsMaxStages = 12;
constexpr uint32_t kTsAcol = 256;   // first TMEM column of the A operand

__global__ void __launch_bounds__(kBmmThreads, 1) a16wfp4_bmm_ts_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                       const BmmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = g.stages, G = g.G;
  uint8_t* xsm = smem;                                        // ring of stages of G x slabs
  uint8_t* osm = xsm + stages * G * kSlabBytes;               // 8 x kStageOutBytes output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(osm + 8 * kStageOutBytes);
  uint64_t* empty = full + kTsMaxStages;
  uint64_t* acc_full = empty + kTsMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x % g.n_tiles;
  const int b = blockIdx.x / g.n_tiles;
  const int mt0 = blockIdx.y * g.m_per_cta;
  const int mt1 = min(g.m_tiles, mt0 + g.m_per_cta);
  bool abort = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kBmmThreads - 64);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- dequantize the weight tile into TMEM (before the dependency wait:
  // the packed weights are never written by the kernel before this one).
  // Warp w stores lanes 32 (w % 4).. (its TMEM quarter), K half (w - 2) / 4;
  // each thread one weight row's 32-element blocks, four in flight.
  if (warp >= 2) {
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int n = nt * 128 + q * 32 + lane;
    const uint8_t* wb = g.w_packed + static_cast<size_t>(b) * g.w_batch_bytes;
    const int nhalf = g.K >> 6;               // 32-element blocks per K half
    const int blk0 = h * nhalf;
    const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + kTsAcol;
    for (int j0 = 0; j0 < nhalf; j0 += 4) {
      uint4 c[4];
      uint32_t sb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j0 + j < nhalf) {
          const int blk = blk0 + j0 + j;
          c[j] = __ldg(reinterpret_cast<const uint4*>(wb + weight_code_offset(n, blk * 16, g.KT)));
          sb[j] = __ldg(wb + weight_scale_offset(n, blk, g.KT));
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j0 + j >= nhalf) break;           // warp-uniform
        const float sc = e8m0_to_float(sb[j]);
        const uint32_t w32[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = dequant_pair((w32[e >> 2] >> (8 * (e & 3))) & 0xFF, sc);
        tmem_st16(ta + static_cast<uint32_t>(blk0 + j0 + j) * 16u, o);
      }
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // x and the output may be written / read by the kernel before this one.
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer: x slabs by TMA, G per stage
      uint32_t ls = 0;
      for (int mt = mt0; mt < mt1; ++mt) {
        for (int ks = 0; ks < g.KS; ks += G, ++ls) {
          const int s = ls % stages;
          const uint32_t ph = (ls / stages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(G * kSlabBytes));
          for (int j = 0; j < G; ++j)
            tma_load_3d(xsm + (s * G + j) * kSlabBytes, &xmap, (ks + j) * 64, mt * 128, b, &full[s]);
        }
        if (abort) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: per slab four 128 x 128 x 16 MMAs, A (weights) from
      // TMEM, B (the x slab) from shared memory; one commit per stage of G
      // slabs (a commit after every four such small MMAs caps the pipe at
      // about one group per 255 ns, sixteen per commit run at 37 ns each).
      const uint32_t idesc = idesc_bf16(128, 128);
      const uint64_t xdesc0 = sdesc_sw128(smem_u32(xsm));
      constexpr uint64_t kSlabStep = kSlabBytes >> 4, kKStep = 32 >> 4;
      int s = 0;
      uint32_t ph = 0;
      int i = 0;
      for (int mt = mt0; mt < mt1 && !abort; ++mt, ++i) {
        const int buf = i & 1;
        const uint32_t use = i >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort)) break;
        tc_fence_after();
        const uint32_t acc = tmem + buf * 128;
        uint32_t acol = tmem + kTsAcol;
        for (int ks = 0; ks < g.KS; ks += G) {
          if (!mbar_wait(&full[s], ph, abort)) break;
          tc_fence_after();
          for (int jg = 0; jg < G; ++jg) {
            const uint64_t xdesc = xdesc0 + static_cast<uint64_t>(s * G + jg) * kSlabStep;
            mma_bf16_ts(acc, acol, xdesc, idesc, (ks + jg) != 0);
#pragma unroll
            for (int j = 1; j < 4; ++j) mma_bf16_ts(acc, acol + j * 8, xdesc + j * kKStep, idesc, 1u);
            acol += 32;
          }
          mma_commit(&empty[s]);
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        mma_commit(&acc_full[buf]);
      }
      // TMEM is freed only after the last drain has read both accumulators.
      for (int k = i - 2 < 0 ? 0 : i - 2; k < i; ++k) mbar_wait(&acc_empty[k & 1], (k >> 1) & 1, abort);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    // ---- epilogue: warp w drains weight rows n0 = 128 nt + 32 (w % 4).. (its
    // lanes) for activation-row columns [64 h, 64 h + 64) in two 32-column
    // pieces.  Lane l holds D[n0 + l][c]; output word (c, i) is the bf16 pair
    // of weight rows n0 + 2i, n0 + 2i + 1 at activation row c, built by lane
    // 2i for even c and lane 2i + 1 for odd c.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint8_t* stg = osm + (warp - 2) * kStageOutBytes;
    const int n0 = nt * 128 + q * 32;
    const int pi = lane >> 1, par = lane & 1;
    auto row_ptr = [&](int m) -> __nv_bfloat16* {
      return g.batch_major ? g.out + (static_cast<size_t>(m) * g.B + b) * g.N
                           : g.out + (static_cast<size_t>(b) * g.M + m) * g.N;
    };
    int i = 0;
    for (int mt = mt0; mt < mt1; ++mt, ++i) {
      const int buf = i & 1;
      const uint32_t use = i >> 1;
      const bool ok = mbar_wait(&acc_full[buf], use & 1, abort);
      tc_fence_after();
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int c0 = h * 64 + p * 32;
        uint32_t r[32];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * 128 + c0,
                  *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * 128 + c0 + 16,
                  *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
        tmem_wait_ld();
        if (p == 1) {
          tc_fence_before();
          mbar_arrive(&acc_empty[buf]);           // this warp's share of the accumulator is read
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t send = par ? r[2 * k] : r[2 * k + 1];
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
          const float lo = __uint_as_float(par ? recv : r[2 * k]);        // weight row n0 + 2 pi
          const float hi = __uint_as_float(par ? r[2 * k + 1] : recv);    // weight row n0 + 2 pi + 1
          *reinterpret_cast<uint32_t*>(stg + (2 * k + par) * 64 + pi * 4) = ok ? pack_bf16x2(lo, hi) : 0u;
        }
        __syncwarp();
#pragma unroll
        for (int pss = 0; pss < 4; ++pss) {
          const int rr = pss * 8 + (lane >> 2), ch = lane & 3;
          const int m = mt * 128 + c0 + rr;
          const int n = n0 + ch * 8;
          const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * 64 + ch * 16);
          if (m < g.M && n < g.N) {
            __nv_bfloat16* dst = row_ptr(m) + n;
            if (g.vec_out && n + 8 <= g.N) {
              *reinterpret_cast<uint4*>(dst) = w;
            } else {
              const uint32_t hw[4] = {w.x, w.y, w.z, w.w};
              for (int e = 0; e < 8 && n + e < g.N; ++e)
                reinterpret_cast<uint16_t*>(dst)[e] = static_cast<uint16_t>(hw[e >> 1] >> (16 * (e & 1)));
            }
          }
        }
        __syncwarp();
      }
    }
  }
  if (abort) atomicOr(&g_bmm_error, kErrTimeout);
}

// ------------------------------------------------------------------ host
// The calling host thread's device context, made current if the runtime has
// not bound it in this thread yet: cuTensorMapEncodeTiled is a driver call
// and runs in the thread's current context, which the runtime binds lazily
// (cudaFree(nullptr) binds it and frees nothing).
static cudaError_t bind_device_context() {
  static thread_local bool bound = false;
  if (bound) return cudaSuccess;
  const cudaError_t e = cudaFree(nullptr);
  if (e == cudaSuccess) bound = true;
  return e;
}

// The driver's tensor-map encoder, looked up once (thread-safe static init).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

static std::atomic<bool> g_bmm_attr[64];      // kernel attribute set on this device
static std::atomic<bool> g_bmm_ts_attr[64];   // the same for a16wfp4_bmm_ts_kernel

cudaError_t launch_bmm(const void* x, const uint8_t* w_packed, void* out, int B, int M, int N, int K,
                       bool batch_major, const DeviceInfo& dev, cudaStream_t s) {
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  cudaError_t ce = bind_device_context();
  if (ce != cudaSuccess) return ce;

  BmmArgs a{};
  a.w_packed = w_packed;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.B = B;
  a.M = M;
  a.N = N;
  a.K = K;
  a.KS = K / 64;
  const int64_t Np = weight_rows(N), Kp = padded_k(K);
  a.KT = static_cast<int>(Kp / kKTile);
  a.w_batch_bytes = static_cast<size_t>(weight_packed_bytes(N, K));
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  // 256 < K <= 512: the weight tile (128 rows) in TMEM, shared memory for x
  const bool ts = K > 256 && K <= 512 && Np % 128 == 0;
  // else the widest weight tile whose bf16 image fits in 128 KiB (and divides Np)
  int BN = ts ? 128 : 256;
  while (BN > 64 && (static_cast<int64_t>(BN) * K * 2 > 128 * 1024 || Np % BN != 0)) BN /= 2;
  a.BN = BN;
  a.n_tiles = static_cast<int>(ceil_div(N, BN));   // tiles holding at least one real weight row
  a.m_tiles = static_cast<int>(ceil_div(M, 128));
  const int pairs = B * a.n_tiles;
  int m_groups = dev.sm_count / pairs;
  if (m_groups < 1) m_groups = 1;
  if (m_groups > a.m_tiles) m_groups = a.m_tiles;
  a.m_per_cta = static_cast<int>(ceil_div(a.m_tiles, m_groups));
  m_groups = static_cast<int>(ceil_div(a.m_tiles, a.m_per_cta));
  a.batch_major = batch_major;
  a.vec_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0 && (N % 8) == 0;

  CUtensorMap map;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(M) * K * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  a.G = 1;
  if (ts) {
    // up to four slabs per ring stage (a divisor of K / 64), one commit each
    const int G = a.KS % 4 == 0 ? 4 : (a.KS % 2 == 0 ? 2 : 1);
    const int fixed_ts = 8 * kStageOutBytes + 1024 + 512;
    int st = (227 * 1024 - fixed_ts) / (G * kSlabBytes);
    if (st > kTsMaxStages / G) st = kTsMaxStages / G;
    a.stages = st;
    a.G = G;
    const int smem_ts = fixed_ts + st * G * kSlabBytes;
    if (!g_bmm_ts_attr[dev.device].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(a16wfp4_bmm_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           227 * 1024);
      if (e != cudaSuccess) return e;
      g_bmm_ts_attr[dev.device].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(pairs), static_cast<unsigned>(m_groups), 1);
    cfg.blockDim = dim3(kBmmThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_ts);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, a16wfp4_bmm_ts_kernel, map, a);
  }

  // x ring: as many 16 KiB slabs as the shared memory left over holds (2..8)
  const int fixed = a.KS * BN * 128 + 8 * kStageOutBytes + 1024 + 256;
  int stages = (227 * 1024 - fixed) / kSlabBytes;
  if (stages > kBmmMaxStages) stages = kBmmMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  a.stages = stages;
  const int smem = fixed + stages * kSlabBytes;
  if (!g_bmm_attr[dev.device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(a16wfp4_bmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    g_bmm_attr[dev.device].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(pairs), static_cast<unsigned>(m_groups), 1);
  cfg.blockDim = dim3(kBmmThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, a16wfp4_bmm_kernel, map, a);
}

uint32_t bmm_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_bmm_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_bmm_error, &zero, sizeof(zero));
  return v;
}

}  // namespace mx
