// Tensor-pipe issue-rate measurement (diagnostic; not on the GEMM path).
//
// One thread per CTA (or per CTA pair) issues the same tcgen05 sequence per
// "step" back to back -- a number of scale copies (shared memory -> TMEM)
// followed by a number of MMAs into one accumulator -- and commits each step
// to a ring of mbarriers, waiting for the commit of the step `depth` back
// before it issues the next: depth 4 is the round trip a 4-stage pipeline
// ring allows, a large depth leaves only the tensor pipe's own throughput.  Operands
// are zero bytes in shared memory: the rates of the tensor pipe do not
// depend on the values.  %globaltimer brackets the timed steps, so each CTA
// reports nanoseconds per step of its own issue stream; launching one CTA
// (or pair) on every SM gives the whole GPU's rate.
//
// The forms are those of the library's kernels: kind::mxf4 block-scaled
// (E2M1 x E2M1, UE8M0 scales, scale_vec::2X, K = 64 per MMA) and kind::f16
// (bf16, K = 16), each with cta_group::1 (M = 128, one SM) or cta_group::2
// (M = 256 over a 2-CTA cluster: each CTA holds its 128 rows of A and half
// of B's N rows; the even CTA issues for both).  Scale copies are
// tcgen05.cp 32x128b.warpx4 (a 512-byte atom replicated into the four lane
// quarters) or 128x256b (4 KiB, no replication).
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_common.cuh"
#include "internal.h"
#include "mxfp4_diag.h"
#include "ptx.cuh"

namespace mx {

constexpr int kRateWarm = 16;                  // untimed steps before the timed ones
constexpr int kRateSmem = 200 * 1024;          // keeps one CTA per SM
constexpr int kRateOperandBytes = 80 * 1024;   // A 16 KiB, B 32 KiB, scale sources 32 KiB
constexpr uint32_t kRateTmemCols = 512;
constexpr int kRateRing = 32;                  // commit barriers; the deepest wait is 32 steps back

struct RateArgs {
  int pair;        // 1: cta_group::2 over a 2-CTA cluster
  int kind;        // 0: kind::mxf4 block-scaled, 1: kind::f16 (bf16)
  int mma_n;       // N of each MMA (M is 128, or 256 for a pair)
  int mmas;        // MMAs per step
  int copies;      // scale copies per step
  int copy_form;   // 0: 32x128b.warpx4, 1: 128x256b
  int steps;       // timed steps
  int depth;       // wait for the commit of the step `depth` back (1..32)
  unsigned long long* ns;   // per unit (CTA or pair): ns of the timed steps, 0 after a timeout
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Descriptor of a 128-row x 32-byte scale source without swizzle: 8-row x
// 16-byte core matrices, the two of a row group 128 bytes apart (leading
// offset), row groups 256 bytes apart (stride offset).
__device__ __forceinline__ uint64_t sdesc_scales_128x256b(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(256 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

template <bool kPair>
__device__ __forceinline__ void rate_copy(int form, uint32_t taddr, uint64_t desc) {
  if (form == 0) {
    if (kPair)
      asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
    else
      asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
  } else {
    if (kPair)
      asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
    else
      asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
  }
}

template <bool kPair>
__device__ __forceinline__ void rate_mma(int kind, uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t sfa,
                                         uint32_t sfb) {
  if (kind == 0) {
    if (kPair)
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
              d),
          "l"(ad), "l"(bd), "r"(id), "r"(sfa), "r"(sfb)
          : "memory");
    else
      mma_mxf4(d, ad, bd, id, sfa, sfb, 1u);
  } else {
    if (kPair)
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
          "l"(ad), "l"(bd), "r"(id)
          : "memory");
    else
      mma_bf16(d, ad, bd, id, 1u);
  }
}

template <bool kPair>
__device__ __forceinline__ void rate_commit(uint64_t* bar) {
  if (kPair)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(static_cast<uint16_t>(3))
        : "memory");
  else
    mma_commit(bar);
}

template <bool kPair>
__global__ void __launch_bounds__(128, 1) tc_rate_kernel(const RateArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  __shared__ uint64_t ring[kRateRing];
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_slot;

  for (int i = threadIdx.x; i < kRateOperandBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();   // the zeros are read by the tensor core (async proxy)
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRateRing; ++s) mbar_init(&ring[s], 1);
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    if (kPair) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                   "r"(kRateTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      tmem_alloc(&tmem_slot, kRateTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync_all();   // both CTAs' barriers and TMEM exist before the first MMA
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool abort = false;
  unsigned long long t0 = 0, t1 = 0;

  if (threadIdx.x == 0 && rank == 0) {
    const uint32_t a_s = smem_u32(smem), b_s = a_s + 16 * 1024, sc_s = a_s + 48 * 1024;
    const int M = kPair ? 256 : 128;
    const int total = kRateWarm + a.steps;
    for (int s = 0; s < total; ++s) {
      const int slot = s & 3;   // scale columns rotate over four slots (their values do not matter)
      if (s >= a.depth) {
        const int w = s - a.depth;
        if (!mbar_wait(&ring[w % kRateRing], static_cast<uint32_t>(w / kRateRing) & 1u, abort)) break;
      }
      tc_fence_after();
      if (s == kRateWarm) t0 = globaltimer();
      const uint32_t scol = tmem + 256u + static_cast<uint32_t>(slot) * 32u;
      for (int c = 0; c < a.copies; ++c) {
        if (a.copy_form == 0)
          rate_copy<kPair>(0, scol + 4u * static_cast<uint32_t>(c & 7), sdesc_scales(sc_s + 512u * (c & 7)));
        else
          rate_copy<kPair>(1, scol + 8u * static_cast<uint32_t>(c & 3),
                           sdesc_scales_128x256b(sc_s + 4096u * (c & 3)));
      }
      for (int j = 0; j < a.mmas; ++j) {
        const uint32_t q = static_cast<uint32_t>(j & 3);
        const uint32_t id = a.kind == 0 ? idesc_mxf4(M, a.mma_n, (q & 1) * 2, (q & 1) * 2) : idesc_bf16(M, a.mma_n);
        rate_mma<kPair>(a.kind, tmem, sdesc_sw128(a_s + 32u * q), sdesc_sw128(b_s + 32u * q), id,
                        scol + 4u * (q >> 1), scol + 16u + 8u * (q >> 1));
      }
      rate_commit<kPair>(&ring[s % kRateRing]);
    }
    // Arrives (in both CTAs of a pair) once every MMA issued above is done.
    rate_commit<kPair>(&done);
  }
  if (threadIdx.x == 0) {
    bool late = false;
    mbar_wait(&done, 0, late);   // bounded; the work above ends in microseconds
    t1 = globaltimer();
    abort = abort || late;
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync_all();   // the pair frees its TMEM together, after its last MMA
  tc_fence_after();
  if (warp == 1) {
    if (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRateTmemCols) : "memory");
    else
      tmem_dealloc(tmem, kRateTmemCols);
  }
  if (threadIdx.x == 0 && rank == 0) a.ns[kPair ? blockIdx.x / 2 : blockIdx.x] = abort ? 0ull : t1 - t0;
}

// Each CTA of a 2-CTA cluster allocates 32 TMEM columns with cta_group::2
// and records the address it got; equal addresses show the allocation is
// one collective operation of the pair.
__global__ void __launch_bounds__(64, 1) tc_pair_alloc_probe_kernel(uint32_t* addr) {
  __shared__ uint32_t slot;
  const uint32_t rank = cluster_ctarank();
  if ((threadIdx.x >> 5) == 0) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&slot)), "r"(32u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) addr[blockIdx.x] = slot | (rank << 30);
  cluster_sync_all();
  if ((threadIdx.x >> 5) == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(slot), "r"(32u) : "memory");
  }
}

static cudaError_t launch_cluster2(const void* kern_tag, int grid, int threads, int smem, cudaStream_t s,
                                   void** args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern_tag, args);
}

}  // namespace mx

using namespace mx;

extern "C" int mxfp4_diag_max_units(void) { return 256; }

extern "C" mxfp4_status mxfp4_diag_pair_alloc_probe(uint32_t* addr_dev, void* stream) {
  if (addr_dev == nullptr) return MXFP4_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess || !dev.ok) return MXFP4_ERR_NO_DEVICE;
  void* args[] = {&addr_dev};
  return launch_cluster2(reinterpret_cast<const void*>(tc_pair_alloc_probe_kernel), 2, 64, 0,
                         static_cast<cudaStream_t>(stream), args) == cudaSuccess
             ? MXFP4_OK
             : MXFP4_ERR_CUDA;
}

extern "C" mxfp4_status mxfp4_diag_tensor_rate(int pair, int kind, int mma_n, int mmas, int copies, int copy_form,
                                               int steps, int depth, unsigned long long* ns_dev, int* units,
                                               void* stream) {
  if (ns_dev == nullptr || units == nullptr) return MXFP4_ERR_INVALID_ARG;
  if ((pair != 0 && pair != 1) || (kind != 0 && kind != 1) || (copy_form != 0 && copy_form != 1))
    return MXFP4_ERR_INVALID_ARG;
  // N: a multiple of 16 in [16, 256] (one CTA), [64, 256] (a pair)
  if (mma_n % 16 != 0 || mma_n > 256 || mma_n < (pair ? 64 : 16)) return MXFP4_ERR_INVALID_ARG;
  if (depth < 1 || depth > kRateRing) return MXFP4_ERR_INVALID_ARG;
  if (mmas < 0 || mmas > 16 || mmas + copies < 1 || copies < 0 || copies > (copy_form == 0 ? 8 : 4) || steps < 1 || steps > 1000000)
    return MXFP4_ERR_INVALID_ARG;
  if (kind == 1 && copies != 0) return MXFP4_ERR_INVALID_ARG;   // bf16 MMAs take no scales
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess || !dev.ok) return MXFP4_ERR_NO_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RateArgs a{pair, kind, mma_n, mmas, copies, copy_form, steps, depth, ns_dev};
  cudaError_t e;
  if (pair == 0) {
    e = cudaFuncSetAttribute(tc_rate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem);
    if (e != cudaSuccess) return MXFP4_ERR_CUDA;
    const int grid = dev.sm_count < mxfp4_diag_max_units() ? dev.sm_count : mxfp4_diag_max_units();
    *units = grid;
    tc_rate_kernel<false><<<grid, 128, kRateSmem, s>>>(a);
    e = cudaGetLastError();
  } else {
    e = cudaFuncSetAttribute(tc_rate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem);
    if (e != cudaSuccess) return MXFP4_ERR_CUDA;
    // as many pairs as the device holds at once, so every pair runs in one wave
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = kRateSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_rate_kernel<true>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = dev.sm_count / 2;
    }
    if (n > dev.sm_count / 2) n = dev.sm_count / 2;
    if (n > mxfp4_diag_max_units()) n = mxfp4_diag_max_units();
    *units = n;
    void* args[] = {&a};
    e = launch_cluster2(reinterpret_cast<const void*>(tc_rate_kernel<true>), 2 * n, 128, kRateSmem, s, args);
  }
  return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}
