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
// kernel is organised to have every SM's copy engine pulling weights from
// the moment it is scheduled until it exits:
//  * stream-K as in the large-M GEMM: output tiles of 128 activation rows
//    (of which only the first 16/32/64 are loaded) by 256 weight rows, the
//    (tile, 256-wide k-step) iterations split evenly over one CTA per SM;
//  * the activation quantization runs inside the kernel: the epilogue warps
//    of CTA c quantize units (k-step, 8 rows) c, c + grid, ... straight into
//    the TILED workspace image and publish a flag per unit; the producer warp
//    requests its first weight stages before anything else and waits for the
//    flags of the k-steps it needs only before their activation copies;
//  * tiles cut by CTA boundaries are summed inside the kernel: every part is
//    published as fp32 with a flag, then each contributing CTA sums a 1/n
//    share of the tile's outputs over all parts in CTA order (deterministic:
//    the same order for every call) and stores them with the bias.
//
// The flags live in the first kDecodeCtrlBytes of the workspace together
// with an epoch word: a call publishes value epoch+1 and waits for exactly
// that value, and the last CTA to finish advances the epoch, so stale flags
// of earlier calls are never mistaken for this call's.  The region must be
// zero before the workspace's first use.
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
  const uint16_t* x;       // bf16 activations [M][ldx], or null when a_codes/a_scales already hold them quantized
  int ldx;
  int vec_ok;              // x and ldx allow 16-byte row loads
  uint8_t* a_codes;        // TILED activation codes (written by this kernel when x != null)
  uint8_t* a_scales;       // TILED activation scales
  const uint8_t* w_codes;
  const uint8_t* w_scales;
  OutView o;
  int M, K, KT;
  int w_tiles;             // Np / 128: 128-row tiles of the packed weights
  int n_tiles;             // ceil(N / 256)
  int total;               // n_tiles x KT iterations
  int grid;
  float* partials;         // 2 slots per CTA, kRowsA x 256 floats each
  uint32_t* ctrl;          // epoch, done counter, part flags, unit flags
};

// Partial-sum slot of CTA c's part of tile t: slot 0 when t is where c's
// range begins, slot 1 when t is where it ends.
__device__ __forceinline__ int part_slot(int c, int t, int KT, int total, int grid) {
  return 2 * c + (sk_begin(c, total, grid) / KT == t ? 0 : 1);
}

template <int kRowsA>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs g) {
  using C = Cfg<kRowsA>;
  constexpr int kGroups = kRowsA / 8;   // 8-row quantization units per k-step
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
  uint32_t* part_flag = g.ctrl + kCtrlPartFlags;
  uint32_t* unit_flag = g.ctrl + kCtrlUnitFlags;
  bool abort = false;
  uint32_t epoch = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiThreads);
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
    auto w_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int t = it / KT, kt = it - t * KT;
      for (int q = 0; q < 2; ++q) {
        const int rt = 2 * t + q;
        if (rt < g.w_tiles) {
          bulk_g2s(st + q * kTileBytes, g.w_codes + (static_cast<size_t>(rt * KT + kt) << 14), kTileBytes, bar);
          bulk_g2s(st + C::kW + C::kA + C::kSA + q * 1024, g.w_scales + (static_cast<size_t>(rt * KT + kt) << 10),
                   1024, bar);
        }
      }
    };
    auto a_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int kt = it % KT;
      bulk_g2s(st + C::kW, g.a_codes + (static_cast<size_t>(kt) << 14), C::kALoad, bar);
      bulk_g2s(st + C::kW + C::kA, g.a_scales + (static_cast<size_t>(kt) << 10), 1024, bar);
    };
    auto stage_bytes = [&](int it) -> uint32_t {
      const int t = it / KT;
      const int nsub = (2 * t + 1 < g.w_tiles) ? 2 : 1;
      return static_cast<uint32_t>(C::kALoad + C::kSA + nsub * (kTileBytes + 1024));
    };
    const int n_iter = it1 - it0;
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
    if (g.x != nullptr) {
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
    abort = __any_sync(0xFFFFFFFFu, abort);
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
          issue_stage_mma<kRowsA>(tmem, smem_u32(smem + s * C::kStageBytes), j != 0 ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        mma_commit(acc_full);
        it += len;
        kt = 0;
      }
    }
    __syncwarp();
  } else {
    griddep_wait();
    epoch = ld_acquire_gpu(g.ctrl + kCtrlEpoch);
    const int et = threadIdx.x - 64;   // 0..255 within the epilogue warps

    // ---- quantize this CTA's activation units: unit u = rg * KT + kt is
    // rows 8 rg .. 8 rg + 7, k-step kt; warp 2 + w takes row 8 rg + w, lane l
    // elements 8 l .. 8 l + 7 of the k-step.  Up to four units per pass have
    // their loads in flight together.
    if (g.x != nullptr) {
      const int units = KT * kGroups;
      const int nb = (g.K + 31) >> 5;
      for (int u0 = cta; u0 < units; u0 += 4 * g.grid) {
        uint16_t v[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int u = u0 + j * g.grid;
          const int kt = u % KT, r = (u / KT) * 8 + (warp - 2);
          load8_bf16(g.x, u < units ? r : g.M, g.M, g.K, g.ldx, kt * 256 + lane * 8, g.vec_ok != 0, v[j]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int u = u0 + j * g.grid;
          if (u >= units) break;   // warp-uniform
          const int kt = u % KT, r = (u / KT) * 8 + (warp - 2);
          uint32_t sbyte;
          const uint32_t packed = quantize8(v[j], sbyte);
          const int blk = kt * 8 + (lane >> 2);
          *reinterpret_cast<uint32_t*>(g.a_codes + tiled_code_offset(r, kt * 128 + lane * 4, KT)) = packed;
          if ((lane & 3) == 0)
            g.a_scales[tiled_scale_offset(r, blk, KT)] = (r < g.M && blk < nb) ? static_cast<uint8_t>(sbyte) : 0x7F;
        }
        // The units are read by other CTAs' bulk copies (async proxy).
        fence_proxy_async_global();
        named_barrier(1, kEpiThreads);
        if (et == 0) {
          __threadfence();
          for (int j = 0; j < 4; ++j) {
            const int u = u0 + j * g.grid;
            if (u < units) st_release_gpu(unit_flag + (u % KT) * 8 + u / KT, epoch + 1);
          }
        }
      }
    }

    // ---- epilogue: warp w drains accumulator rows 32*(w%4).., columns 128*h..
    const OutView& o = g.o;
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int rl = q * 32 + lane;                 // accumulator row = activation row
    const bool warp_live = q * 32 < kRowsA;       // quarters beyond kRowsA rows hold nothing
    const bool live = warp_live && rl < g.M;
    int split_first = -1, split_last = -1;        // this CTA's tiles that other CTAs share
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
        float v[64];
        if (warp_live) {
          uint32_t r[64];
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16)
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + pass * 64 + c0,
                      *reinterpret_cast<uint32_t(*)[16]>(&r[c0]));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 64; ++c) v[c] = ok ? __uint_as_float(r[c]) : 0.f;
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
            for (int c = 0; c < 32; ++c) chunk[c] = v[c0 + c];
            store_chunk(o, rl, n0 + pass * 64 + c0, chunk);
          }
        } else {
          float4* P = reinterpret_cast<float4*>(g.partials + (static_cast<size_t>(slot) * kRowsA + rl) * kTileN +
                                                h * 128 + pass * 64);
#pragma unroll
          for (int c = 0; c < 16; ++c) __stcg(P + c, make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
        }
      }
      if (!whole) {
        named_barrier(1, kEpiThreads);          // the whole part is written
        if (et == 0) {
          __threadfence();
          st_release_gpu(part_flag + slot, epoch + 1);
        }
        if (it == it0) split_first = t;
        else split_last = t;
      }
      it += len;
      kt = 0;
    }

    // ---- shared tiles: contributor j of n sums outputs [j/n, (j+1)/n) of
    // the tile over every part in CTA order, adds the bias, stores bf16.
    // Each thread keeps 2 groups (4 consecutive outputs each) x 4 parts of
    // loads in flight.
    for (int which = 0; which < 2; ++which) {
      const int t = which == 0 ? split_first : split_last;
      if (t < 0) continue;
      const int c_lo = sk_owner(t * KT, g.total, g.grid);
      const int c_hi = sk_owner(t * KT + KT - 1, g.total, g.grid);
      if (warp == 2) {
        for (int c = c_lo + lane; c <= c_hi; c += 32)
          if (c != cta) flag_wait(part_flag + part_slot(c, t, KT, g.total, g.grid), epoch + 1, abort);
      }
      named_barrier(1, kEpiThreads);
      const int n_c = c_hi - c_lo + 1;
      const int groups = g.M * (kTileN / 4);
      const int j = cta - c_lo;
      const int gb = static_cast<int>(static_cast<long long>(j) * groups / n_c);
      const int ge = static_cast<int>(static_cast<long long>(j + 1) * groups / n_c);
      for (int g0 = gb + et; g0 < ge; g0 += 2 * kEpiThreads) {
        float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        for (int cg = c_lo; cg <= c_hi; cg += 4) {
          float4 p[4][2];
#pragma unroll
          for (int jc = 0; jc < 4; ++jc) {
            const int cc = cg + jc;
            if (cc > c_hi) continue;
            const float4* Q = reinterpret_cast<const float4*>(
                g.partials + static_cast<size_t>(part_slot(cc, t, KT, g.total, g.grid)) * kRowsA * kTileN);
#pragma unroll
            for (int k = 0; k < 2; ++k)
              if (g0 + kEpiThreads * k < ge) p[jc][k] = __ldcg(Q + g0 + kEpiThreads * k);
          }
#pragma unroll
          for (int jc = 0; jc < 4; ++jc) {
            if (cg + jc > c_hi) continue;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              acc[k].x += p[jc][k].x;
              acc[k].y += p[jc][k].y;
              acc[k].z += p[jc][k].z;
              acc[k].w += p[jc][k].w;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int gi = g0 + kEpiThreads * k;
          if (gi < ge) store_quad(o, gi / (kTileN / 4), t * kTileN + 4 * (gi % (kTileN / 4)), acc[k]);
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
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<kRowsA>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    g_attr_set[dev.device][which] = true;
  }
  return launch_pdl(decode_kernel<kRowsA>, a.grid, kThreads, C::kSmem, s, a);
}

cudaError_t launch_decode(const DecodeProblem& p, const DeviceInfo& dev, cudaStream_t s) {
  DecodeArgs a{};
  const int64_t Np = padded_rows(p.N);
  const int64_t Kp = padded_k(p.K);
  a.x = static_cast<const uint16_t*>(p.x);
  a.ldx = p.ldx;
  a.vec_ok = p.x != nullptr && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.ldx % 8) == 0;
  a.a_codes = const_cast<uint8_t*>(p.a_codes);
  a.a_scales = const_cast<uint8_t*>(p.a_scales);
  a.w_codes = p.w_packed;
  a.w_scales = p.w_packed + Np * Kp / 2;
  a.o.out = static_cast<__nv_bfloat16*>(p.out);
  a.o.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.o.ldo = p.ldo;
  a.o.N = p.N;
  a.M = p.M;
  a.K = p.K;
  a.KT = static_cast<int>(Kp / kKTile);
  a.w_tiles = static_cast<int>(Np / 128);
  a.n_tiles = static_cast<int>(ceil_div(p.N, kTileN));
  a.total = a.n_tiles * a.KT;
  int grid = gemm_grid(dev);
  if (grid > a.total) grid = a.total;
  a.grid = grid;
  a.partials = p.partials;
  a.ctrl = p.ctrl;
  if (p.x != nullptr && a.KT > kMaxFusedKT) return cudaErrorInvalidValue;
  switch (gemm_rows_a(p.M)) {
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
