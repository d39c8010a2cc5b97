// W4A4 MXFP4 GEMM for decode-sized activations (M <= 64): the whole linear
// layer -- activation quantization, GEMM, split-tile reduction, bias and
// bf16 store -- in one kernel launch.
//
//   out[m][n] = bf16_RNE( sum_k deq(Q(x))[m][k] * deq(W)[n][k] + bias[n] )
//
// the per_1x32_f4_quant + gemm_a4w4 + bias steps of sglang PR #39598 (blog
// analysis, section 2, apply_weights), for the small-M shapes whose cost is
// streaming the packed weights once.
//
// At M <= 64 the weights are almost all of the bytes (N*K/2 codes against
// 2*M*K activation bytes), and a call lasts only a few microseconds, so the
// kernel is organised around one dependent chain per call (activations ready
// -> MMAs -> split-tile sums -> outputs) with as much of the weight stream as
// possible taken off it:
//  * output tiles of 128 activation rows (of which only the first 16/32/64
//    are loaded) by 256 weight rows; with fewer tiles than SMs every tile is
//    split into the same number of k-ranges, one CTA each (an even stream-K
//    split of the (tile, 256-wide k-step) iterations whose parts line up with
//    tile boundaries), which leaves the remaining SMs free for the next
//    launch to start on;
//  * the kernel is a programmatic dependent launch and lets its own
//    dependent launch at once, so a CTA requests its first weight stages as
//    soon as it has an SM, usually while the previous call is still running
//    (the packed weights are never written by the kernel this one follows);
//  * the activations are quantized inside the kernel: every CTA quantizes a
//    share of the (k-step, 8-row) units into the workspace (blocked form) and
//    publishes a flag per unit, and producers copy a k-step in once its
//    units are flagged;
//  * tiles cut by CTA boundaries are summed inside the kernel: every part is
//    published as fp32 with a flag, then each contributing CTA sums a 1/n
//    share of the tile's outputs over all parts in CTA order (deterministic:
//    the same order for every call) and stores them with the bias.
//
// The part flags live in the first kDecodeCtrlBytes of the workspace with an
// epoch word: a call publishes value epoch+1 and waits for exactly that
// value, and the last CTA to finish advances the epoch, so stale flags of
// earlier calls are never mistaken for this call's.  The region must be zero
// before the workspace's first use.
//
// Every CTA must be resident at the same time (a CTA waits for flags that
// other CTAs set).  The grid is at most one CTA per SM and a CTA's shared
// memory exceeds half of an SM's, so this holds as soon as the kernels ahead
// of it drain; every wait is bounded and records kErrTimeout instead of
// hanging if another stream keeps SMs occupied for longer than that bound.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_common.cuh"
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {

static __device__ uint32_t g_decode_error;

struct DecodeArgs {
  const uint16_t* x;       // bf16 activations [M][ldx] (mode kQuantGlobal)
  int ldx;
  int vec_ok;              // x and ldx allow 16-byte row loads
  int mode;                // kPrequantized or kQuantGlobal
  uint8_t* a_codes;        // TILED codes, or blocked activations (a_blocked; kRowsA-row blocks)
  uint8_t* a_scales;       // TILED activation scales (unused when a_blocked)
  int a_blocked;           // set when the kernel or the quantizer wrote the blocked form
  const uint8_t* w_packed;         // packed weight blocks
  OutView o;
  int M, K, KT;
  int n_tiles;             // ceil(N / 256)
  int total;               // n_tiles x KT iterations
  int grid;
  float* partials;         // 2 slots per CTA, kRowsA x 256 floats each
  uint32_t* ctrl;          // epoch, done counter, part flags
};

// Loads this lane's 8 bf16 values of row r, elements [e0, e0 + 8), as a
// uint4 (zeros past K or for r >= M).
__device__ __forceinline__ uint4 load8_packed(const uint16_t* __restrict__ x, int r, int M, int K, int ldx, int e0,
                                              bool vec_ok) {
  if (r >= M) return make_uint4(0, 0, 0, 0);
  const uint16_t* src = x + static_cast<size_t>(r) * ldx + e0;
  if (vec_ok && e0 + 8 <= K) return __ldg(reinterpret_cast<const uint4*>(src));
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = e0 + 2 * i < K ? src[2 * i] : 0u;
    const uint32_t hi = e0 + 2 * i + 1 < K ? src[2 * i + 1] : 0u;
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Where the activation codes of a stage come from.
//  kPrequantized: the caller's TILED codes/scales, copied in by the producer.
//  kQuantGlobal:  every CTA first quantizes a share of the (k-step, 8-row)
//                 units into the workspace (blocked form) and publishes a flag
//                 per unit; producers wait for the flags of their k-steps and
//                 copy the codes in.  x is read once in all.
// (Quantizing inside each CTA from its own copy of x was measured slower at
// every M: its stages complete at a fraction of the rate of copied ones.)
enum DecodeMode : int { kPrequantized = 0, kQuantGlobal = 1 };

// Partial-sum slot of CTA c's part of tile t: slot 0 when t is where c's
// range begins, slot 1 when t is where it ends.
__device__ __forceinline__ int part_slot(int c, int t, int KT, int total, int grid) {
  return 2 * c + (sk_begin(c, total, grid) / KT == t ? 0 : 1);
}

constexpr int kDrainThreads = 128;     // warps 4, 5, 8, 9: accumulator rows 0..63
// Named barriers (0 is __syncthreads).
constexpr uint32_t kBarDrain = 2, kBarAll = 3;

template <int kRowsA>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs g) {
  using C = Cfg<kRowsA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRing);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = g.KT;
  const int cta = blockIdx.x;
  const int it0 = sk_begin(cta, g.total, g.grid);
  const int it1 = sk_begin(cta + 1, g.total, g.grid);
  const int n_iter = it1 - it0;
  uint32_t* part_flag = g.ctrl + kCtrlPartFlags;
  uint32_t* unit_flag = g.ctrl + kCtrlUnitFlags;
  constexpr int kGroups = kRowsA / 8;         // 8-row quantization units per k-step (kQuantGlobal)
  bool abort = false;
  uint32_t epoch = 0;

  // Tiles of this range shared with other CTAs: the first segment when the
  // range starts inside a tile or ends before that tile's end, the last one
  // when the range ends inside a later tile (CTA-uniform).
  const int t_first = it0 / KT, t_last = (it1 - 1) / KT;
  const int split_first = (it0 % KT != 0 || it1 < (t_first + 1) * KT) ? t_first : -1;
  const int split_last = (t_last != t_first && it1 % KT != 0) ? t_last : -1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kDrainThreads);
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
  // The next kernel in the stream waits for this one to complete before it
  // touches memory, so it may be launched now; its CTAs take SMs as this
  // kernel's CTAs leave.
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ---- producer.  A stage is one 256-wide k-step of one output tile.
    // Weights are read once: evict-first keeps L2 for the activations and
    // the partial sums.
    const uint64_t evict_first = policy_evict_first();
    auto w_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int t = it / KT, kt = it - t * KT;
      bulk_g2s_hint(st, g.w_packed + static_cast<size_t>(t * KT + kt) * kWeightBlockBytes, kWeightBlockBytes, bar,
                    evict_first);
    };
    // Activations of the stage's k-step (rows 0..kRowsA-1 of row tile 0):
    // one copy of the blocked form, or codes + scales of the TILED form.
    auto a_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int kt = it % KT;
      if (g.a_blocked) {
        bulk_g2s(st + C::kW, g.a_codes + static_cast<size_t>(kt) * (C::kALoad + C::kSA), C::kALoad + C::kSA, bar);
      } else {
        bulk_g2s(st + C::kW, g.a_codes + (static_cast<size_t>(kt) << 14), C::kALoad, bar);
        bulk_g2s(st + C::kW + C::kA, g.a_scales + (static_cast<size_t>(kt) << 10), 1024, bar);
      }
    };
    auto stage_bytes = [&](int) -> uint32_t { return static_cast<uint32_t>(C::kW + C::kALoad + C::kSA); };
    const int npre = n_iter < C::kStages ? n_iter : C::kStages;
    // Lane i requests the weights of prologue stage i at once: the packed
    // weights are never written by the kernel this one follows (the repack
    // ends with an ordinary launch).
    if (lane < npre) {
      mbar_arrive_expect_tx(&full[lane], stage_bytes(it0 + lane));
      w_load(it0 + lane, smem + lane * C::kStageBytes, &full[lane]);
    }
    griddep_wait();
    epoch = ld_acquire_gpu(g.ctrl + kCtrlEpoch);
    if (g.mode == kQuantGlobal) {
      // Wait until every activation k-step this CTA reads is quantized: the
      // lanes share the (k-step, 8-row unit) flags of the range.
      const int nkt = n_iter < KT ? n_iter : KT;
      const int kt_first = it0 % KT;
      for (int idx = lane; idx < nkt * kGroups; idx += 32) {
        int kt = kt_first + idx / kGroups;
        if (kt >= KT) kt -= KT;
        flag_wait(unit_flag + kt * 8 + idx % kGroups, epoch + 1, abort);
      }
      __syncwarp();                  // every lane is ordered after every lane's acquire
      fence_proxy_async_global();    // ... and so are its bulk copies below
    }
    if (lane < npre) a_load(it0 + lane, smem + lane * C::kStageBytes, &full[lane]);
    __syncwarp();
    if (lane == 0) {
      for (int i = npre; i < n_iter; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes(it0 + i));
        w_load(it0 + i, st, &full[s]);
        a_load(it0 + i, st, &full[s]);
      }
    }
    __syncwarp();   // whole warp reaches the final barrier converged
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: one accumulator, one segment (part of a tile) at a time
      int i = 0, seg = 0, kt = it0 % KT;
      for (int it = it0; it < it1 && !abort; ++seg) {
        const int len = (KT - kt) < (it1 - it) ? (KT - kt) : (it1 - it);
        if (!mbar_wait(acc_empty, (seg & 1) ^ 1, abort)) break;
        tc_fence_after();
        for (int j = 0; j < len; ++j, ++i) {
          const int s = i % C::kStages;
          const uint32_t ph = (i / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, abort)) break;
          tc_fence_after();
          issue_stage_mma<C>(tmem, smem_u32(smem + s * C::kStageBytes), j != 0 ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        mma_commit(acc_full);
        it += len;
        kt = 0;
      }
    }
    __syncwarp();
  } else {
    // ---- warps 2..9
    const int et = threadIdx.x - 64;   // 0..255
    if (g.mode == kQuantGlobal && g.vec_ok != 0 && lane == 0) {
      // L2 prefetch of the rows of this CTA's first units (a prefetch returns
      // no data, so it may run before the dependency wait).
      const int units = KT * kGroups;
      for (int u = cta; u < units && u < cta + 4 * g.grid; u += g.grid) {
        const int kt = u % KT, r = (u / KT) * 8 + (warp - 2);
        const int n = g.K - kt * 256 < 256 ? g.K - kt * 256 : 256;
        const uint32_t bytes = static_cast<uint32_t>(2 * n) & ~15u;
        if (r < g.M && bytes != 0) bulk_prefetch_l2(g.x + static_cast<size_t>(r) * g.ldx + kt * 256, bytes);
      }
    }
    if (g.mode == kQuantGlobal) {
      griddep_wait();
      epoch = ld_acquire_gpu(g.ctrl + kCtrlEpoch);
      // Quantize this CTA's units into the workspace (blocked form): unit
      // u = rg * KT + kt is rows 8 rg .. 8 rg + 7 of k-step kt; warp 2 + w
      // takes row 8 rg + w, lane l elements 8 l .. 8 l + 7.  Up to four units
      // per pass have their loads in flight together.
      const int units = KT * kGroups;
      const int nb = (g.K + 31) >> 5;
      for (int u0 = cta; u0 < units; u0 += 4 * g.grid) {
        uint4 v4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int u = u0 + j * g.grid;
          const int kt = u % KT, r = (u / KT) * 8 + (warp - 2);
          v4[j] = load8_packed(g.x, u < units ? r : g.M, g.M, g.K, g.ldx, kt * 256 + lane * 8, g.vec_ok != 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int u = u0 + j * g.grid;
          if (u >= units) break;   // warp-uniform
          const int kt = u % KT, r = (u / KT) * 8 + (warp - 2);
          const uint16_t v[8] = {static_cast<uint16_t>(v4[j].x & 0xFFFF), static_cast<uint16_t>(v4[j].x >> 16),
                                 static_cast<uint16_t>(v4[j].y & 0xFFFF), static_cast<uint16_t>(v4[j].y >> 16),
                                 static_cast<uint16_t>(v4[j].z & 0xFFFF), static_cast<uint16_t>(v4[j].z >> 16),
                                 static_cast<uint16_t>(v4[j].w & 0xFFFF), static_cast<uint16_t>(v4[j].w >> 16)};
          uint32_t sbyte;
          const uint32_t packed = quantize8(v, sbyte);
          const int blk = kt * 8 + (lane >> 2);
          *reinterpret_cast<uint32_t*>(g.a_codes + blocked_code_offset(r, kt * 128 + lane * 4, KT, kRowsA)) = packed;
          if ((lane & 3) == 0)
            g.a_codes[blocked_scale_offset(r, blk, KT, kRowsA)] =
                (r < g.M && blk < nb) ? static_cast<uint8_t>(sbyte) : 0x7F;
        }
        // The units are read by other CTAs' bulk copies (async proxy).
        fence_proxy_async_global();
        named_barrier(kBarAll, kEpiThreads);
        if (et == 0) {
          for (int j = 0; j < 4; ++j) {
            const int u = u0 + j * g.grid;
            if (u < units) st_release_gpu(unit_flag + (u % KT) * 8 + u / KT, epoch + 1);
          }
        }
      }
    }
  if ((warp & 3) >= 2) {
    // ---- warps 2, 3, 6, 7: idle until the shared-tile sums.
    griddep_wait();
    if (g.mode != kQuantGlobal) epoch = ld_acquire_gpu(g.ctrl + kCtrlEpoch);
  } else {
    // ---- warps 4, 5, 8, 9 drain the accumulator: warp w rows 32 (w % 4)..,
    // columns 128 h.. (h = 0 for warps 4, 5; 1 for 8, 9).
    if (g.mode != kQuantGlobal) {
      griddep_wait();
      epoch = ld_acquire_gpu(g.ctrl + kCtrlEpoch);
    }
    const OutView& o = g.o;
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int rl = q * 32 + lane;                 // accumulator row = activation row
    const bool live = rl < g.M;
    int seg = 0, kt = it0 % KT;
    for (int it = it0; it < it1; ++seg) {
      const int len = (KT - kt) < (it1 - it) ? (KT - kt) : (it1 - it);
      const int t = it / KT;
      const bool ok = mbar_wait(acc_full, seg & 1, abort);
      tc_fence_after();
      const int n0 = t * kTileN + h * 128;
      const bool whole = kt == 0 && len == KT;
      const int slot = 2 * cta + (it == it0 ? 0 : 1);
      // Two passes of 64 columns; the accumulator is released right after the
      // second pass is loaded.  A whole tile is stored; a part is published.
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t r[64];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16)
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + pass * 64 + c0,
                    *reinterpret_cast<uint32_t(*)[16]>(&r[c0]));
        tmem_wait_ld();
        if (!ok) {
#pragma unroll
          for (int c = 0; c < 64; ++c) r[c] = 0u;
        }
        if (pass == 1) {
          tc_fence_before();
          mbar_arrive(acc_empty);
        }
        if (!live) continue;
        if (whole) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            float chunk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) chunk[c] = __uint_as_float(r[c0 + c]);
            store_chunk(o, rl, n0 + pass * 64 + c0, chunk);
          }
        } else {
          uint4* P = reinterpret_cast<uint4*>(g.partials + (static_cast<size_t>(slot) * kRowsA + rl) * kTileN +
                                              h * 128 + pass * 64);
#pragma unroll
          for (int c = 0; c < 16; ++c) __stcg(P + c, make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]));
        }
      }
      if (!whole) {
        named_barrier(kBarDrain, kDrainThreads);       // the whole part is written
        if (threadIdx.x == 128) st_release_gpu(part_flag + slot, epoch + 1);
      }
      it += len;
      kt = 0;
    }
  }
  }

  // ---- shared tiles (at most two), by warps 2..9.  Contributor j of n
  // finishes outputs [j/n, (j+1)/n) of the tile: warp 2 waits for the other
  // parts, then each thread sums 4 groups (4 consecutive outputs each) over
  // all parts in CTA order, 4 parts' loads in flight per group, adds the bias
  // and stores bf16.
  if (warp >= 2 && (split_first >= 0 || split_last >= 0)) {
    const int et = threadIdx.x - 64;   // 0..255
    const int groups = g.M * (kTileN / 4);     // float4 groups of a tile's live rows
    if (warp == 2) {
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int t = w == 0 ? split_first : split_last;
        if (t < 0) continue;
        const int lo = sk_owner(t * KT, g.total, g.grid), hi = sk_owner(t * KT + KT - 1, g.total, g.grid);
        for (int c = lo + lane; c <= hi; c += 32)
          if (c != cta) flag_wait(part_flag + part_slot(c, t, KT, g.total, g.grid), epoch + 1, abort);
      }
    }
    named_barrier(kBarAll, kEpiThreads);
#pragma unroll 1
    for (int w = 0; w < 2; ++w) {
      const int t = w == 0 ? split_first : split_last;
      if (t < 0) continue;
      const int lo = sk_owner(t * KT, g.total, g.grid);
      const int nc = sk_owner(t * KT + KT - 1, g.total, g.grid) - lo + 1;
      const int j = cta - lo;
      const int gb = static_cast<int>(static_cast<long long>(j) * groups / nc);
      const int ge = static_cast<int>(static_cast<long long>(j + 1) * groups / nc);
      for (int g0 = gb + et; g0 < ge; g0 += 4 * kEpiThreads) {
        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int cg = 0; cg < nc; cg += 4) {
          float4 p[4][4];
#pragma unroll
          for (int jc = 0; jc < 4; ++jc) {
            if (cg + jc >= nc) continue;
            const float4* Q = reinterpret_cast<const float4*>(
                g.partials + static_cast<size_t>(part_slot(lo + cg + jc, t, KT, g.total, g.grid)) * kRowsA * kTileN);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (g0 + k * kEpiThreads < ge) p[k][jc] = __ldcg(Q + g0 + k * kEpiThreads);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int jc = 0; jc < 4; ++jc) {
              if (cg + jc >= nc) continue;
              acc[k].x += p[k][jc].x;
              acc[k].y += p[k][jc].y;
              acc[k].z += p[k][jc].z;
              acc[k].w += p[k][jc].w;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int gi = g0 + k * kEpiThreads;
          if (gi < ge) store_quad(g.o, gi / (kTileN / 4), t * kTileN + 4 * (gi % (kTileN / 4)), acc[k]);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (abort) atomicOr(&g_decode_error, kErrTimeout);
  // The last CTA out advances the epoch: every CTA has read it by then, and
  // the next call reads it only after this grid has completed.
  if (threadIdx.x == 0) {
    const uint32_t done = atomicInc(g.ctrl + kCtrlDone, static_cast<unsigned>(g.grid - 1));
    if (done == static_cast<uint32_t>(g.grid - 1)) {
      __threadfence();
      st_release_gpu(g.ctrl + kCtrlEpoch, epoch + 1);
    }
  }
}

// ===================================================================== host
static bool g_attr_set[64][3];

template <int kRowsA>
static cudaError_t launch_rows(const DecodeArgs& a, const DeviceInfo& dev, cudaStream_t s, int which) {
  using C = Cfg<kRowsA>;
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev.device][which]) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<kRowsA>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    g_attr_set[dev.device][which] = true;
  }
  return launch_pdl(decode_kernel<kRowsA>, a.grid, kThreads, C::kSmem, s, a);
}

cudaError_t launch_decode(const DecodeProblem& p, const DeviceInfo& dev, cudaStream_t s) {
  DecodeArgs a{};
  const int64_t Kp = padded_k(p.K);
  a.x = static_cast<const uint16_t*>(p.x);
  a.ldx = p.ldx;
  a.vec_ok = p.x != nullptr && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.ldx % 8) == 0;
  a.a_codes = const_cast<uint8_t*>(p.a_codes);
  a.a_scales = const_cast<uint8_t*>(p.a_scales);
  a.w_packed = p.w_packed;
  a.o.out = static_cast<__nv_bfloat16*>(p.out);
  a.o.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.o.ldo = p.ldo;
  a.o.N = p.N;
  a.M = p.M;
  a.K = p.K;
  a.KT = static_cast<int>(Kp / kKTile);
  a.n_tiles = static_cast<int>(ceil_div(p.N, kTileN));
  a.total = a.n_tiles * a.KT;
  // With fewer 256-row tiles than SMs, split every tile into the same number
  // S of k-ranges (grid = tiles x S): each CTA then works on one tile, parts
  // line up with tile boundaries (S parts per tile when S divides K/256), and
  // the SMs left over are free for the next launch to start on.  More tiles
  // than SMs: balanced stream-K over all SMs.
  const int max_grid = gemm_grid(dev);
  int grid = max_grid;
  if (a.n_tiles < max_grid) {
    int split = max_grid / a.n_tiles;
    if (split > a.KT) split = a.KT;
    grid = a.n_tiles * split;
  }
  if (grid > a.total) grid = a.total;
  a.grid = grid;
  a.partials = p.partials;
  a.ctrl = p.ctrl;
  // Activation source: copied in when pre-quantized; else quantized by all
  // CTAs with unit flags; past the flags' K range, by the standalone
  // quantizer kernel first.
  const int rows = gemm_rows_a(p.M);
  if (p.x == nullptr) {
    a.mode = kPrequantized;            // the caller's TILED codes and scales
    a.a_blocked = 0;
  } else if (a.KT <= kMaxUnitKT) {
    a.mode = kQuantGlobal;             // blocked form, written by this kernel
    a.a_blocked = 1;
  } else {
    cudaError_t e = launch_quant(p.x, p.M, p.K, p.ldx, a.a_codes, nullptr, ActLayout::kBlocked, rows, dev, s);
    if (e != cudaSuccess) return e;
    a.mode = kPrequantized;
    a.a_blocked = 1;
  }
  switch (rows) {
    case 16: return launch_rows<16>(a, dev, s, 0);
    case 32: return launch_rows<32>(a, dev, s, 1);
    default: return launch_rows<64>(a, dev, s, 2);
  }
}

uint32_t decode_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero));
  return v;
}

}  // namespace mx
