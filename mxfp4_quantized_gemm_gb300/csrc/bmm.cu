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
// every warp store writes whole 64-byte row segments.  The kernel is a
// programmatic dependent launch: the weight tile is dequantized before the
// wait for the kernel ahead of it.
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
  int stages;                // x ring depth
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

// ------------------------------------------------------------------ host
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

static std::atomic<bool> g_bmm_attr[64];   // kernel attribute set on this device

cudaError_t launch_bmm(const void* x, const uint8_t* w_packed, void* out, int B, int M, int N, int K,
                       bool batch_major, const DeviceInfo& dev, cudaStream_t s) {
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;

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
  // widest weight tile whose bf16 image fits in 128 KiB (and divides Np)
  int BN = 256;
  while (BN > 64 && (static_cast<int64_t>(BN) * K * 2 > 128 * 1024 || Np % BN != 0)) BN /= 2;
  a.BN = BN;
  a.n_tiles = static_cast<int>(Np / BN);
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

  // x ring: as many 16 KiB slabs as the shared memory left over holds (2..8)
  const int fixed = a.KS * BN * 128 + 8 * kStageOutBytes + 1024 + 256;
  int stages = (227 * 1024 - fixed) / kSlabBytes;
  if (stages > kBmmMaxStages) stages = kBmmMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  a.stages = stages;
  const int smem = fixed + stages * kSlabBytes;
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
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
