// Tensor-pipe issue-rate measurement (diagnostic; not on the GEMM path).
//
// One thread per CTA (or per CTA pair; or two threads per CTA, each with its
// own accumulator) issues the same tcgen05 sequence per "step" back to back -- a number of scale copies (shared memory -> TMEM)
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
constexpr int kRateRing = 128;                 // commit barriers: 32 steps back of up to 4 commits each

struct RateArgs {
  int mma_n;       // N of each MMA (M is 128, or 256 for a pair)
  int steps;       // timed steps
  int depth;       // wait for the commit of the step `depth` back (1..32)
  unsigned long long* ns;   // per unit (CTA or pair): ns of the timed steps, 0 after a timeout
};

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

template <bool kPair, int kForm>
__device__ __forceinline__ void rate_copy(uint32_t taddr, uint64_t desc) {
  if (kForm == 0) {
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

template <bool kPair, int kKind>
__device__ __forceinline__ void rate_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t sfa,
                                         uint32_t sfb) {
  if (kKind == 2) {
    // the same block-scaled E2M1 product (UE8M0 scales, one per 32 elements)
    // issued as kind::mxf4nvf4
    if (kPair)
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
              "r"(d),
          "l"(ad), "l"(bd), "r"(id), "r"(sfa), "r"(sfb)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
              "r"(d),
          "l"(ad), "l"(bd), "r"(id), "r"(sfa), "r"(sfb)
          : "memory");
  } else if (kKind == 0) {
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

// One instruction mix, fully unrolled: kMmas MMAs of kind kKind (0: mxf4,
// 1: bf16, 2: the mxf4 product issued as kind::mxf4nvf4) and kCopies scale
// copies of form kForm per step (groups of four MMAs, each after its share
// of the copies), issued by
// kIssuers threads of the CTA (lane 0 of warps 0 and 1), each into its own
// accumulator (columns 0.. and 128.. ; N <= 128 with two issuers) and its
// own scale columns (256.. and 384..).
template <bool kPair, int kKind, int kMmas, int kCopies, int kForm, int kIssuers, int kMode>
__global__ void __launch_bounds__(128, 1) tc_rate_kernel(const RateArgs a) {
  constexpr int kGroups = kMmas >= 4 ? kMmas / 4 : 1;
  constexpr bool kSplitCommit = kMode == 1;
  constexpr int kCommits = kSplitCommit ? kGroups : 1;   // commits per step
  constexpr int kMmasPerGroup = kMmas >= 4 ? 4 : kMmas;
  static_assert(kCopies % kGroups == 0, "copies split evenly over the groups of four MMAs");
  static_assert(32 * kCommits <= kRateRing, "the deepest wait's commit still has its own barrier");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  __shared__ uint64_t ring[kIssuers][kRateRing];
  __shared__ uint64_t done[kIssuers];
  __shared__ uint32_t tmem_slot;

  for (int i = threadIdx.x; i < kRateOperandBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();   // the zeros are read by the tensor core (async proxy)
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kIssuers; ++w) {
      for (int s = 0; s < kRateRing; ++s) mbar_init(&ring[w][s], 1);
      mbar_init(&done[w], 1);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
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

  const int issuer = warp;   // lane 0 of warps 0 .. kIssuers-1
  if ((threadIdx.x & 31) == 0 && issuer < kIssuers && rank == 0) {
    const uint32_t a_s = smem_u32(smem), b_s = a_s + 16 * 1024, sc_s = a_s + 48 * 1024;
    constexpr int M = kPair ? 256 : 128;
    const uint32_t dcol = tmem + 128u * static_cast<uint32_t>(issuer);
    const uint32_t scbase = tmem + 256u + 128u * static_cast<uint32_t>(issuer);
    const int total = kRateWarm + a.steps;
    uint32_t id[2];
    for (int h = 0; h < 2; ++h) id[h] = kKind != 1 ? idesc_mxf4(M, a.mma_n, h * 2, h * 2) : idesc_bf16(M, a.mma_n);
    for (int s = 0; s < total; ++s) {
      if (s >= a.depth) {
        const int w = (s - a.depth) * kCommits + kCommits - 1;   // the last commit of that step
        if (!mbar_wait(&ring[issuer][w % kRateRing], static_cast<uint32_t>(w / kRateRing) & 1u, abort)) break;
      }
      tc_fence_after();
      if (s == kRateWarm) t0 = globaltimer();
      const uint32_t scol = scbase + static_cast<uint32_t>(s & 3) * 32u;   // four rotating slots (values unused)
      // In groups of four MMAs (a 256-wide k-step of the GEMMs), each after
      // its share of the step's copies and one commit per step; or
      // (kSplitCommit) every group's copies first, then each group's MMAs
      // followed by a commit of its own.
#pragma unroll
      for (int grp = 0; grp < kGroups; ++grp) {
#pragma unroll
        for (int c0 = 0; c0 < (kSplitCommit ? kCopies : kCopies / kGroups); ++c0) {
          if (kSplitCommit && grp != 0) break;
          const int c = kSplitCommit ? c0 : grp * (kCopies / kGroups) + c0;
          if (kForm == 0)
            rate_copy<kPair, 0>(scol + 4u * (c & 7), sdesc_scales(sc_s + 512u * (c & 7)));
          else
            rate_copy<kPair, 1>(scol + 8u * (c & 3), sdesc_scales_128x256b(sc_s + 4096u * (c & 3)));
        }
        // kMode 2: the previous step's commit between this step's copies and
        // its MMAs, so that no copy directly follows a commit
        if (kMode == 2 && grp == 0 && s > 0) rate_commit<kPair>(&ring[issuer][(s - 1) % kRateRing]);
#pragma unroll
        for (int j = 0; j < kMmasPerGroup; ++j) {
          const uint32_t q = static_cast<uint32_t>(j & 3);
          rate_mma<kPair, kKind>(dcol, sdesc_sw128(a_s + 32u * q), sdesc_sw128(b_s + 32u * q), id[q & 1],
                                 scol + 4u * (q >> 1), scol + 16u + 8u * (q >> 1));
        }
        if (kSplitCommit) {
          const int c = s * kCommits + grp;
          rate_commit<kPair>(&ring[issuer][c % kRateRing]);
        }
      }
      if (kMode == 0) rate_commit<kPair>(&ring[issuer][s % kRateRing]);
    }
    if (kMode == 2 && total > 0 && !abort) rate_commit<kPair>(&ring[issuer][(total - 1) % kRateRing]);
    // Arrives (in both CTAs of a pair) once every instruction issued above is done.
    rate_commit<kPair>(&done[issuer]);
  }
  if ((threadIdx.x & 31) == 0 && issuer < kIssuers) {
    bool late = false;
    mbar_wait(&done[issuer], 0, late);   // bounded; the work above ends in microseconds
    t1 = globaltimer();
    abort = abort || late;
  }
  __shared__ unsigned long long span[kIssuers];
  if ((threadIdx.x & 31) == 0 && issuer < kIssuers) span[issuer] = abort ? 0ull : t1 - t0;
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync_all();   // the pair frees its TMEM together, after its last MMA
  tc_fence_after();
  if (warp == 2) {
    if (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRateTmemCols) : "memory");
    else
      tmem_dealloc(tmem, kRateTmemCols);
  }
  if (threadIdx.x == 0 && rank == 0) {
    unsigned long long worst = 0;
    bool any_zero = false;
    for (int w = 0; w < kIssuers; ++w) {
      worst = span[w] > worst ? span[w] : worst;
      any_zero = any_zero || span[w] == 0;
    }
    a.ns[kPair ? blockIdx.x / 2 : blockIdx.x] = any_zero ? 0ull : worst;
  }
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

namespace mx {

// The measured instruction mixes: pair, kind, MMAs and scale copies per
// step, copy form, issuing threads, commit placement (0: after the step's
// MMAs; 1: the step's copies all first, a commit after every group of four
// MMAs; 2: the step's commit deferred past the next step's copies).
struct RateVariant {
  int pair, kind, mmas, copies, form, issuers, split;   // split: the commit placement
  void* kernel;
};
#define MX_RATE(P, K, MM, C, F, I) \
  { P, K, MM, C, F, I, 0, reinterpret_cast<void*>(tc_rate_kernel<P != 0, K, MM, C, F, I, 0>) }
#define MX_RATE_MODE(MM, C, F, MODE) \
  { 0, 0, MM, C, F, 1, MODE, reinterpret_cast<void*>(tc_rate_kernel<false, 0, MM, C, F, 1, MODE>) }
static const RateVariant kRateVariants[] = {
    MX_RATE(0, 0, 4, 0, 0, 1),  MX_RATE(0, 0, 4, 6, 0, 1),  MX_RATE(0, 0, 4, 4, 0, 1),
    MX_RATE(0, 0, 4, 2, 1, 1),  MX_RATE(0, 0, 8, 0, 0, 1),  MX_RATE(0, 0, 16, 0, 0, 1),
    MX_RATE(0, 0, 0, 6, 0, 1),  MX_RATE(0, 0, 4, 0, 0, 2),  MX_RATE(0, 0, 4, 4, 0, 2),
    MX_RATE(0, 0, 16, 0, 0, 2), MX_RATE(1, 0, 4, 0, 0, 1),  MX_RATE(1, 0, 4, 6, 0, 1),
    MX_RATE(1, 0, 4, 4, 0, 1),  MX_RATE(1, 0, 16, 0, 0, 1), MX_RATE(0, 1, 4, 0, 0, 1),
    MX_RATE(1, 1, 4, 0, 0, 1),  MX_RATE(0, 1, 16, 0, 0, 1), MX_RATE(0, 1, 16, 0, 0, 2),
    MX_RATE(0, 2, 16, 0, 0, 1), MX_RATE(0, 2, 4, 4, 0, 1),  MX_RATE(1, 2, 16, 0, 0, 1),
    // several k-steps per commit
    MX_RATE(0, 0, 8, 8, 0, 1),  MX_RATE(0, 0, 16, 16, 0, 1), MX_RATE(0, 0, 8, 4, 1, 1),
    MX_RATE(0, 0, 8, 12, 0, 1), MX_RATE(0, 1, 8, 0, 0, 1),
    // copies of two or four k-steps issued ahead, a commit after each k-step's MMAs
    MX_RATE_MODE(8, 8, 0, 1),   MX_RATE_MODE(16, 16, 0, 1), MX_RATE_MODE(8, 12, 0, 1),
    MX_RATE_MODE(8, 4, 1, 1),
    // each step's commit deferred past the next step's copies
    MX_RATE_MODE(4, 4, 0, 2),   MX_RATE_MODE(4, 6, 0, 2),   MX_RATE_MODE(4, 2, 1, 2),
};
#undef MX_RATE
#undef MX_RATE_MODE
constexpr int kNumRateVariants = static_cast<int>(sizeof(kRateVariants) / sizeof(kRateVariants[0]));

}  // namespace mx

extern "C" int mxfp4_diag_tensor_rate_variants(void) { return mx::kNumRateVariants; }

extern "C" mxfp4_status mxfp4_diag_tensor_rate_info(int variant, int* info) {
  if (variant < 0 || variant >= mx::kNumRateVariants || info == nullptr) return MXFP4_ERR_INVALID_ARG;
  const mx::RateVariant& v = mx::kRateVariants[variant];
  info[0] = v.pair;
  info[1] = v.kind;
  info[2] = v.mmas;
  info[3] = v.copies;
  info[4] = v.form;
  info[5] = v.issuers;
  info[6] = v.split;
  return MXFP4_OK;
}

extern "C" mxfp4_status mxfp4_diag_tensor_rate(int variant, int mma_n, int steps, int depth,
                                               unsigned long long* ns_dev, int* units, void* stream) {
  if (ns_dev == nullptr || units == nullptr || variant < 0 || variant >= kNumRateVariants)
    return MXFP4_ERR_INVALID_ARG;
  const RateVariant& v = kRateVariants[variant];
  // N: a multiple of 16 in [16, 256] (one CTA), [64, 256] (a pair), at most 128 with two issuers
  if (mma_n % 16 != 0 || mma_n > (v.issuers == 2 ? 128 : 256) || mma_n < (v.pair ? 64 : 16))
    return MXFP4_ERR_INVALID_ARG;
  // a deferred commit (placement 2) is issued one step late: waiting on the step just before
  // would wait on a commit not yet issued
  if (steps < 1 || steps > 1000000 || depth < (v.split == 2 ? 2 : 1) || depth > 32) return MXFP4_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess || !dev.ok) return MXFP4_ERR_NO_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RateArgs a{mma_n, steps, depth, ns_dev};
  void* args[] = {&a};
  cudaError_t e = cudaFuncSetAttribute(v.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem);
  if (e != cudaSuccess) return MXFP4_ERR_CUDA;
  if (v.pair == 0) {
    const int grid = dev.sm_count < mxfp4_diag_max_units() ? dev.sm_count : mxfp4_diag_max_units();
    *units = grid;
    e = cudaLaunchKernel(v.kernel, dim3(grid), dim3(128), args, kRateSmem, s);
  } else {
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
    if (cudaOccupancyMaxActiveClusters(&n, v.kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = dev.sm_count / 2;
    }
    if (n > dev.sm_count / 2) n = dev.sm_count / 2;
    if (n > mxfp4_diag_max_units()) n = mxfp4_diag_max_units();
    *units = n;
    e = launch_cluster2(v.kernel, 2 * n, 128, kRateSmem, s, args);
  }
  return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}
