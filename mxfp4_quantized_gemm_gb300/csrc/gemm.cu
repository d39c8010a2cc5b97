// W4A4 MXFP4 GEMM on the sm_103a block-scaled tensor cores.
//
//   out[m][n] = bf16_RNE( sum_k deq(A)[m][k] * deq(W)[n][k] + bias[n] )
//
// the gemm_a4w4 + bias step of sglang PR #39598 (blog analysis, section 2,
// apply_weights).  Both operands arrive in the TILED layout, so every stage
// is a handful of contiguous 1-D bulk copies (16 KiB code tiles already in
// the 128-byte-swizzled K-major image, 512-byte scale atoms already in the
// tcgen05.cp source layout).  One thread issues
// tcgen05.mma.kind::mxf4.block_scale (K = 64 per instruction, two UE8M0
// scales per row per instruction) into a TMEM fp32 accumulator; four warps
// drain TMEM with tcgen05.ld and run the bias + bf16 epilogue.
//
// Two kernels share that machinery:
//  * prefill (M > 64): one CTA per 128 x 256 output tile, full K;
//  * decode (M <= 64): swap-AB -- the weight rows are the MMA's M = 128
//    operand and the few activation rows its N (16/32/64) -- with a balanced
//    stream-K split of the (weight tile, k-tile) iteration space over one CTA
//    per SM, so every SM streams the same number of weight bytes; partial
//    tiles are summed by the last CTA to finish them (atomic ticket, fixed
//    summation order, no waiting).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mx {

static __device__ uint32_t g_gemm_error;

struct GemmArgs {
  const uint8_t* a_codes;
  const uint8_t* a_scales;
  const uint8_t* w_codes;
  const uint8_t* w_scales;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  int ldo, M, N, KT;
  int w_tiles;          // Np / 128
  // stream-K (decode)
  float* partials;
  unsigned long long* tickets;   // per weight tile: (call tag << 16) | arrivals
  unsigned long long tag;        // 48-bit tag of this call
  int grid;
  int64_t total_iters;
};

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// ===================================================================== prefill
constexpr int kPfBN = 256;
constexpr int kPfStages = 4;
constexpr int kPfA = kTileBytes;                     // 128 rows of A codes
constexpr int kPfB = kPfBN * 128;                    // 256 rows of W codes
constexpr int kPfSA = 1024;                          // 2 scale atoms of A
constexpr int kPfSB = (kPfBN / 128) * 1024;          // 2 x 2 scale atoms of W
constexpr int kPfStageBytes = kPfA + kPfB + kPfSA + kPfSB;
constexpr int kPfSmem = kPfStages * kPfStageBytes + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kPfTmemCols = 512;                // 256 accumulator + 24 scale columns

__global__ void __launch_bounds__(192, 1) gemm_prefill_kernel(const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPfStages * kPfStageBytes);
  uint64_t* empty = full + kPfStages;
  uint64_t* done = empty + kPfStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, mt = blockIdx.y;
  const int KT = g.KT;
  bool abort = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kPfTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer: bulk copies of one k-tile per stage.  The weight tiles
      // of the first stages are requested before waiting on the kernel that
      // produces the activations (programmatic dependent launch).
      const int nsub = min(2, g.w_tiles - nt * 2);   // weight row tiles that exist
      const uint32_t bytes = kPfA + kPfSA + nsub * (kTileBytes + 1024);
      auto load_w = [&](int kt, uint8_t* st, uint64_t* bar) {
        for (int q = 0; q < nsub; ++q) {
          const int rt = nt * 2 + q;
          bulk_g2s(st + kPfA + q * kTileBytes, g.w_codes + (static_cast<size_t>(rt * KT + kt) << 14), kTileBytes, bar);
          bulk_g2s(st + kPfA + kPfB + kPfSA + q * 1024, g.w_scales + (static_cast<size_t>(rt * 2 * KT + 2 * kt) << 9),
                   1024, bar);
        }
      };
      auto load_a = [&](int kt, uint8_t* st, uint64_t* bar) {
        bulk_g2s(st, g.a_codes + (static_cast<size_t>(mt * KT + kt) << 14), kTileBytes, bar);
        bulk_g2s(st + kPfA + kPfB, g.a_scales + (static_cast<size_t>(mt * 2 * KT + 2 * kt) << 9), 1024, bar);
      };
      const int npre = min(kPfStages, KT);
      for (int kt = 0; kt < npre; ++kt) {
        mbar_arrive_expect_tx(&full[kt], bytes);
        load_w(kt, smem + kt * kPfStageBytes, &full[kt]);
      }
      griddep_wait();
      for (int kt = 0; kt < npre; ++kt) load_a(kt, smem + kt * kPfStageBytes, &full[kt]);
      for (int kt = npre; kt < KT; ++kt) {
        const int s = kt % kPfStages;
        const uint32_t ph = (kt / kPfStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
        uint8_t* st = smem + s * kPfStageBytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        load_w(kt, st, &full[s]);
        load_a(kt, st, &full[s]);
      }
    }
    __syncwarp();   // whole warp reaches the final barrier converged
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      const uint32_t acc = tmem;
      const uint32_t sfa = tmem + 256;       // 2 atoms x 4 columns
      const uint32_t sfb = tmem + 264;       // 2 atoms x (2 row groups x 4 columns)
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % kPfStages;
        const uint32_t ph = (kt / kPfStages) & 1;
        if (!mbar_wait(&full[s], ph, abort)) break;
        tc_fence_after();
        const uint32_t base = smem_u32(smem + s * kPfStageBytes);
        const uint32_t a_s = base, b_s = base + kPfA, sa_s = base + kPfA + kPfB, sb_s = sa_s + kPfSA;
        tmem_cp_scales(sfa + 0, sdesc_scales(sa_s));
        tmem_cp_scales(sfa + 4, sdesc_scales(sa_s + 512));
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int q = 0; q < 2; ++q) tmem_cp_scales(sfb + a * 8 + q * 4, sdesc_scales(sb_s + q * 1024 + a * 512));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t id = idesc_mxf4(128, kPfBN, (j & 1) * 2, (j & 1) * 2);
          mma_mxf4(acc, sdesc_sw128(a_s + 32 * j), sdesc_sw128(b_s + 32 * j), id, sfa + 4 * (j >> 1),
                   sfb + 8 * (j >> 1), (kt | j) != 0);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(done);
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM -> registers -> + bias -> bf16 -> global
    griddep_wait();
    const bool ok = mbar_wait(done, 0, abort);
    tc_fence_after();
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = mt * 128 + q * 32 + lane;
    if (ok) {
#pragma unroll 1
      for (int c0 = 0; c0 < kPfBN; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
        tmem_wait_ld();
        const int n0 = nt * kPfBN + c0;
        if (row < g.M && n0 < g.N) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            v[i] = __uint_as_float(r[i]);
            if (g.bias != nullptr && n0 + i < g.N)
              v[i] += bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(g.bias) + n0 + i));
          }
          __nv_bfloat16* dst = g.out + static_cast<size_t>(row) * g.ldo + n0;
          if (n0 + 16 <= g.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            uint4 w0, w1;
            w0.x = pack_bf16x2(v[0], v[1]);   w0.y = pack_bf16x2(v[2], v[3]);
            w0.z = pack_bf16x2(v[4], v[5]);   w0.w = pack_bf16x2(v[6], v[7]);
            w1.x = pack_bf16x2(v[8], v[9]);   w1.y = pack_bf16x2(v[10], v[11]);
            w1.z = pack_bf16x2(v[12], v[13]); w1.w = pack_bf16x2(v[14], v[15]);
            reinterpret_cast<uint4*>(dst)[0] = w0;
            reinterpret_cast<uint4*>(dst)[1] = w1;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (n0 + i < g.N) dst[i] = __float2bfloat16_rn(v[i]);
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPfTmemCols);
  }
  if (abort) atomicOr(&g_gemm_error, kErrTimeout);
}

// ===================================================================== decode
template <int BN>
struct DecodeCfg {
  static constexpr int kW = kTileBytes;          // 128 weight rows
  static constexpr int kSW = 1024;               // 2 weight scale atoms
  static constexpr int kA = BN * 128;            // BN activation rows
  static constexpr int kSA = 1024;               // 2 activation scale atoms
  static constexpr int kStageBytes = kW + kSW + kA + kSA;
  static constexpr int kStages = (200 * 1024) / kStageBytes > 10 ? 10 : (200 * 1024) / kStageBytes;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 512;
  static constexpr uint32_t kAccCols = 2 * BN;   // double-buffered accumulator
  static constexpr uint32_t kTmemCols = (kAccCols + 16 <= 64) ? 64 : (kAccCols + 16 <= 128) ? 128 : 256;
};

__device__ __forceinline__ int64_t sk_begin(int c, int64_t total, int grid) {
  return (static_cast<int64_t>(c) * total) / grid;
}
// CTA whose balanced range [sk_begin(c), sk_begin(c+1)) holds iteration `it`.
__device__ __forceinline__ int sk_owner(int64_t it, int64_t total, int grid) {
  int c = static_cast<int>((it * grid) / total);
  while (c + 1 < grid && sk_begin(c + 1, total, grid) <= it) ++c;
  while (c > 0 && sk_begin(c, total, grid) > it) --c;
  return c;
}

// End (exclusive k-tile) of the segment that starts at k-tile ka of a tile
// when `left` iterations of the CTA's range remain.
__device__ __forceinline__ int64_t seg_end(int KT, int ka, int64_t left) {
  const int64_t e = ka + left;
  return e < KT ? e : KT;
}

template <int BN>
__global__ void __launch_bounds__(192, 1) gemm_decode_kernel(const GemmArgs g) {
  using C = DecodeCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile uint32_t* last_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = g.KT;
  const int cta = blockIdx.x;
  const int64_t it0 = sk_begin(cta, g.total_iters, g.grid);
  const int64_t it1 = sk_begin(cta + 1, g.total_iters, g.grid);
  bool abort = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer.  Weight tiles of the first stages are requested before
      // waiting on the activation-producing kernel (programmatic dependent launch).
      const uint32_t bytes = C::kStageBytes;
      auto load_w = [&](int64_t it, uint8_t* st, uint64_t* bar) {
        const int t = static_cast<int>(it / KT);
        const int kt = static_cast<int>(it - static_cast<int64_t>(t) * KT);
        bulk_g2s(st, g.w_codes + (static_cast<size_t>(t * KT + kt) << 14), kTileBytes, bar);
        bulk_g2s(st + C::kW, g.w_scales + (static_cast<size_t>(t * 2 * KT + 2 * kt) << 9), 1024, bar);
      };
      auto load_a = [&](int64_t it, uint8_t* st, uint64_t* bar) {
        const int kt = static_cast<int>(it % KT);
        bulk_g2s(st + C::kW + C::kSW, g.a_codes + (static_cast<size_t>(kt) << 14), C::kA, bar);
        bulk_g2s(st + C::kW + C::kSW + C::kA, g.a_scales + (static_cast<size_t>(2 * kt) << 9), 1024, bar);
      };
      const int npre = static_cast<int>((it1 - it0) < C::kStages ? (it1 - it0) : C::kStages);
      for (int i = 0; i < npre; ++i) {
        mbar_arrive_expect_tx(&full[i], bytes);
        load_w(it0 + i, smem + i * C::kStageBytes, &full[i]);
      }
      griddep_wait();
      for (int i = 0; i < npre; ++i) load_a(it0 + i, smem + i * C::kStageBytes, &full[i]);
      uint32_t ls = npre;
      for (int64_t it = it0 + npre; it < it1; ++it, ++ls) {
        const int s = ls % C::kStages;
        const uint32_t ph = (ls / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        load_w(it, st, &full[s]);
        load_a(it, st, &full[s]);
      }
    }
    __syncwarp();   // whole warp reaches the final barrier converged
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: one accumulator per tile segment, double-buffered
      const uint32_t sfa = tmem + C::kAccCols;
      const uint32_t sfb = tmem + C::kAccCols + 8;
      uint32_t ls = 0;
      int seg = 0;
      for (int64_t it = it0; it < it1 && !abort; ++seg) {
        const int t = static_cast<int>(it / KT);
        const int ka = static_cast<int>(it - static_cast<int64_t>(t) * KT);
        const int kb = static_cast<int>(seg_end(KT, ka, it1 - it));
        const int buf = seg & 1;
        const uint32_t use = seg >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort)) break;
        tc_fence_after();
        const uint32_t acc = tmem + buf * BN;
        for (int kt = ka; kt < kb; ++kt, ++ls) {
          const int s = ls % C::kStages;
          const uint32_t ph = (ls / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, abort)) break;
          tc_fence_after();
          const uint32_t base = smem_u32(smem + s * C::kStageBytes);
          const uint32_t w_s = base, sw_s = base + C::kW, a_s = sw_s + C::kSW, sa_s = a_s + C::kA;
          tmem_cp_scales(sfa + 0, sdesc_scales(sw_s));
          tmem_cp_scales(sfa + 4, sdesc_scales(sw_s + 512));
          tmem_cp_scales(sfb + 0, sdesc_scales(sa_s));
          tmem_cp_scales(sfb + 4, sdesc_scales(sa_s + 512));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t id = idesc_mxf4(128, BN, (j & 1) * 2, (j & 1) * 2);
            mma_mxf4(acc, sdesc_sw128(w_s + 32 * j), sdesc_sw128(a_s + 32 * j), id, sfa + 4 * (j >> 1),
                     sfb + 4 * (j >> 1), (kt != ka || j != 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full[buf]);
        it += kb - ka;
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue (128 threads): lane = weight row n, columns = activation rows m
    griddep_wait();
    const int q = warp & 3;
    const int rl = q * 32 + lane;            // row inside the 128-row weight tile
    int seg = 0;
    for (int64_t it = it0; it < it1; ++seg) {
      const int t = static_cast<int>(it / KT);
      const int ka = static_cast<int>(it - static_cast<int64_t>(t) * KT);
      const int kb = static_cast<int>(seg_end(KT, ka, it1 - it));
      const int buf = seg & 1;
      const uint32_t use = seg >> 1;
      const bool ok = mbar_wait(&acc_full[buf], use & 1, abort);
      tc_fence_after();
      float v[BN];
      if (ok) {
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + c0, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[c0 + i] = __uint_as_float(r[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < BN; ++i) v[i] = 0.f;
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);

      const int n = t * 128 + rl;
      const float b = (g.bias != nullptr && n < g.N)
                          ? bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(g.bias) + n))
                          : 0.f;
      const bool whole = (ka == 0 && kb == KT);
      if (whole) {
        if (n < g.N) {
#pragma unroll
          for (int m = 0; m < BN; ++m)
            if (m < g.M) g.out[static_cast<size_t>(m) * g.ldo + n] = __float2bfloat16_rn(v[m] + b);
        }
      } else {
        // partial tile: publish the fp32 partial, last finisher sums in order
        const int slot = 2 * cta + (it == it0 ? 0 : 1);
        float* P = g.partials + static_cast<size_t>(slot) * (BN * 128);
#pragma unroll
        for (int m = 0; m < BN; ++m) __stcg(P + m * 128 + rl, v[m]);
        __threadfence();
        named_barrier(1, 128);
        const int64_t tb = static_cast<int64_t>(t) * KT;
        const int c_lo = sk_owner(tb, g.total_iters, g.grid);
        const int c_hi = sk_owner(tb + KT - 1, g.total_iters, g.grid);
        if (threadIdx.x == 64) {
          // Arrival count of this call on tile t.  A word whose tag is not this
          // call's counts as zero, so the workspace needs no initialisation.
          unsigned long long* tk = &g.tickets[t];
          unsigned long long cur = atomicAdd(tk, 0ull);
          unsigned long long before;
          while (true) {
            before = ((cur >> 16) == g.tag) ? (cur & 0xFFFFull) : 0ull;
            const unsigned long long want = (g.tag << 16) | (before + 1);
            const unsigned long long seen = atomicCAS(tk, cur, want);
            if (seen == cur) break;
            cur = seen;
          }
          *last_flag = (before == static_cast<unsigned long long>(c_hi - c_lo)) ? 1u : 0u;
        }
        named_barrier(1, 128);
        if (*last_flag) {
          __threadfence();
          float sum[BN];
#pragma unroll
          for (int m = 0; m < BN; ++m) sum[m] = 0.f;
          for (int cc = c_lo; cc <= c_hi; ++cc) {
            const int64_t b0 = sk_begin(cc, g.total_iters, g.grid);
            const int sl = 2 * cc + ((b0 / KT) == t ? 0 : 1);
            const float* Q = g.partials + static_cast<size_t>(sl) * (BN * 128);
#pragma unroll
            for (int m = 0; m < BN; ++m)
              if (m < g.M) sum[m] += __ldcg(Q + m * 128 + rl);
          }
          if (n < g.N) {
#pragma unroll
            for (int m = 0; m < BN; ++m)
              if (m < g.M) g.out[static_cast<size_t>(m) * g.ldo + n] = __float2bfloat16_rn(sum[m] + b);
          }
          if (threadIdx.x == 64) atomicExch(&g.tickets[t], 0ull);   // leave the ticket clean
        }
        named_barrier(1, 128);
      }
      it += kb - ka;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (abort) atomicOr(&g_gemm_error, kErrTimeout);
}

// ===================================================================== host
static bool g_attr_set[64][4];

template <typename Kern>
static cudaError_t ensure_smem(Kern k, int smem, int dev, int which) {
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev][which]) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    g_attr_set[dev][which] = true;
  }
  return cudaSuccess;
}

size_t gemm_streamk_workspace_bytes(int M, int N, int K) {
  (void)M;
  (void)K;
  const size_t partials = static_cast<size_t>(2) * kMaxStreamKCtas * kDecodeMaxM * 128 * sizeof(float);
  const size_t tickets = static_cast<size_t>(ceil_div(N, 128)) * sizeof(unsigned long long);
  return partials + ((tickets + 255) & ~static_cast<size_t>(255));
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream (the activation quantizer) is finishing;
// it waits on it with griddepcontrol.wait before reading activations.
template <typename Kern>
static cudaError_t launch_pdl(Kern k, dim3 grid, int smem, cudaStream_t s, const GemmArgs& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

template <int BN>
static cudaError_t launch_decode(GemmArgs& a, const DeviceInfo& dev, cudaStream_t s, int which) {
  using C = DecodeCfg<BN>;
  cudaError_t e = ensure_smem(gemm_decode_kernel<BN>, C::kSmem, dev.device, which);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_decode_kernel<BN>, dim3(a.grid), C::kSmem, s, a);
}

// 48-bit tag distinguishing this call's stream-K tickets from stale words.
static unsigned long long next_call_tag() {
  static std::atomic<unsigned long long> seq{0};
  unsigned long long x = seq.fetch_add(1, std::memory_order_relaxed) + 0x632BE59BD9B4E019ull;
  x ^= x >> 31;
  x *= 0x9E3779B97F4A7C15ull;
  x ^= x >> 29;
  x &= 0xFFFFFFFFFFFFull;
  return x == 0 ? 1 : x;
}

cudaError_t launch_gemm(const GemmProblem& p, const DeviceInfo& dev, cudaStream_t s) {
  GemmArgs a{};
  const int64_t Np = padded_rows(p.N);
  const int64_t Kp = padded_k(p.K);
  a.a_codes = p.a_codes;
  a.a_scales = p.a_scales;
  a.w_codes = p.w_packed;
  a.w_scales = p.w_packed + Np * Kp / 2;
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.ldo = p.ldo;
  a.M = p.M;
  a.N = p.N;
  a.KT = static_cast<int>(Kp / kKTile);
  a.w_tiles = static_cast<int>(Np / 128);

  if (p.M <= kDecodeMaxM) {
    a.total_iters = static_cast<int64_t>(a.w_tiles) * a.KT;
    int grid = dev.sm_count < kMaxStreamKCtas ? dev.sm_count : kMaxStreamKCtas;
    if (grid > a.total_iters) grid = static_cast<int>(a.total_iters);
    a.grid = grid;
    a.partials = static_cast<float*>(p.workspace);
    const size_t partial_bytes = static_cast<size_t>(2) * kMaxStreamKCtas * kDecodeMaxM * 128 * sizeof(float);
    a.tickets = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(p.workspace) + partial_bytes);
    a.tag = next_call_tag();
    if (p.M <= 16) return launch_decode<16>(a, dev, s, 1);
    if (p.M <= 32) return launch_decode<32>(a, dev, s, 2);
    return launch_decode<64>(a, dev, s, 3);
  }
  cudaError_t e = ensure_smem(gemm_prefill_kernel, kPfSmem, dev.device, 0);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(ceil_div(p.N, kPfBN)), static_cast<unsigned>(ceil_div(p.M, 128)));
  return launch_pdl(gemm_prefill_kernel, grid, kPfSmem, s, a);
}

uint32_t gemm_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
  return v;
}

}  // namespace mx
