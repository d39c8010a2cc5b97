// W4A4 MXFP4 GEMM for decode-sized activations (M <= 64): the linear layer
// -- activation quantization (for M <= 8; above that the quantizer kernel
// runs first), GEMM, split-K reduction, bias and bf16 store -- in one kernel
// launch.
//
//   out[m][n] = bf16_RNE( sum_k deq(Q(x))[m][k] * deq(W)[n][k] + bias[n] )
//
// the per_1x32_f4_quant + gemm_a4w4 + bias steps of sglang PR #39598 (blog
// analysis, section 2, apply_weights), for the small-M shapes whose cost is
// streaming the packed weights once.
//
// At M <= 64 the weights are almost all of the bytes (N*K/2 codes against
// 2*M*K activation bytes) and a call lasts a few microseconds, so the kernel
// is built around a short dependent chain per call with the weight stream
// taken off it:
//  * output tiles of 128 activation rows (only the first M are live) by 256
//    weight rows, one tcgen05 block-scaled MMA accumulator per tile;
//  * with fewer tiles than SMs every tile is split into S k-ranges, one CTA
//    each, and the S CTAs of a tile form a thread-block cluster: each CTA
//    leaves its fp32 partial tile in its own shared memory and, after one
//    cluster barrier, sums a 1/S column share of all S partials through
//    distributed shared memory (in rank order, so the result is the same
//    for every call), adds the bias and stores bf16.  No CTA ever waits for
//    a CTA outside its cluster, and the kernel needs no global scratch;
//  * with at least as many tiles as SMs (S = 1) each CTA takes whole tiles;
//  * the kernel is a programmatic dependent launch and lets its own
//    dependent launch at once: a CTA requests its first weight stages as soon
//    as it has an SM, usually while the previous call is still running (the
//    packed weights are never written by the kernel this one follows);
//  * for M <= 8 every CTA quantizes the activations of its own k-steps
//    straight into the operand slots of its stages (one row per warp, its x
//    loads several stages ahead), so the MMAs start one L2 round trip after
//    the dependency wait; for larger M (where every CTA re-reading bf16 x
//    would cost as much L2 traffic as its weights) the standalone quantizer
//    runs first and the kernel copies the quantized rows in with one bulk
//    copy per stage;
//  * decode_kernel<rows, true> is the MXFP4 output epilogue's form (the
//    results quantized per 1x32 along N instead of stored as bf16); the bf16
//    form is a separate instantiation that holds none of that code.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm_common.cuh"
#include "internal.h"
#include "layout.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {

static __device__ uint32_t g_decode_error;

// Timeline stamps (built only with -DMXFP4_STAMPS, the library's timeline
// variant): %globaltimer at fixed points of every CTA of the last
// kStampCalls launches, for the per-call timeline the benchmark prints.
#ifdef MXFP4_STAMPS
constexpr int kStampCalls = 64, kStampCtas = 256, kStampPoints = 8;
// point 0 of each CTA's row holds the launch's sequence number in its top 16
// bits (the timer's low 48 bits hold ~78 hours of nanoseconds), so rows
// left from an older launch in the same slot can be told apart
static __device__ unsigned long long g_stamps[kStampCalls][kStampCtas][kStampPoints];
__device__ __forceinline__ void stamp_at(int seq, int point) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  if (point == 0) t = (t & 0xFFFFFFFFFFFFull) | (static_cast<unsigned long long>(seq & 0xFFFF) << 48);
  if (blockIdx.x < kStampCtas) g_stamps[seq % kStampCalls][blockIdx.x][point] = t;
}
#define MX_STAMP(p) stamp_at(g.stamp_call, p)
#else
#define MX_STAMP(p) ((void)0)
#endif

struct DecodeArgs {
  const uint16_t* x;       // bf16 activations [M][ldx], quantized in the kernel; null: a_codes/a_scales
  int ldx;
  int vec_ok;              // x and ldx allow 16-byte row loads
  const uint8_t* a_codes;  // x == null: TILED activation codes, or the blocked activations (a_blocked)
  const uint8_t* a_scales; // x == null: TILED activation scales (unused when a_blocked)
  int a_blocked;           // a_codes holds blocked activations (kRowsA-row blocks)
  const uint8_t* w_packed; // packed weight blocks
  OutView o;
  int M, K, KT;
  int n_tiles;             // ceil(N / 256)
  int split;               // CTAs per tile = cluster size; 1: CTAs take whole tiles
#ifdef MXFP4_STAMPS
  int stamp_call;          // slot of this launch in the stamp buffer
#endif
};

constexpr int kLoadAhead = 8;        // x loads in flight per quantizing warp
constexpr int kDrainThreads = 128;   // warps 4, 5, 8, 9: accumulator rows 0..63

// Byte offset of the 16-byte chunk q (4 fp32 columns) of partial-tile row r
// in a CTA's shared memory: 1 KiB per row, chunks XOR-swizzled by r % 8 so a
// warp's rows spread over all banks.
__device__ __forceinline__ uint32_t partial_off(int r, int q) {
  return static_cast<uint32_t>(r) * 1024u + ((static_cast<uint32_t>(q) ^ (r & 7)) << 4);
}

// MXFP4 output of a split tile (the cluster sum's other form): the CTA of
// rank `rank` takes 32-column blocks [8 rank / S, 8 (rank + 1) / S); 8
// consecutive lanes share one (row, block), lane `sub` summing its 4 columns
// 4 sub.. over the S parts in rank order (the sums of the bf16 path, in the
// same order), and quantize it together.  Whole warps loop, so every lane
// takes part in the shuffles.  Called by warps 2..9.
__device__ __forceinline__ void split_sum_store_q(const OutView o, int M, int S, int rank, uint32_t pbase, int n0) {
  const int b_lo = rank * 8 / S, nbk = (rank + 1) * 8 / S - b_lo;
  const int total = M * nbk * 8;
  const int lane = threadIdx.x & 31;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(o.bias);
  for (int base = (threadIdx.x - 64) & ~31; base < total; base += kEpiThreads) {
    const int gi = base + lane;
    const bool act = gi < total;
    const int unit = gi >> 3, sub = gi & 7;
    const int r = act ? unit / nbk : 0, bb = b_lo + (act ? unit % nbk : 0);
    const int n = n0 + 32 * bb + 4 * sub;      // this lane's first column
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (act) {
      const uint32_t a = pbase + partial_off(r, bb * 8 + sub);
      float4 p[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < S) p[k] = ld_shared_cluster_f4(mapa_shared(a, static_cast<uint32_t>(k)));
      acc = p[0];
#pragma unroll
      for (int k = 1; k < 8; ++k) {
        if (k < S) {
          acc.x += p[k].x;
          acc.y += p[k].y;
          acc.z += p[k].z;
          acc.w += p[k].w;
        }
      }
    }
    // + bias and bf16 as store_quad forms them; columns past N are zeros
    float x[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = act && n + i < o.N ? with_bias(bias, n + i, x[i]) : 0.f;
    const uint32_t w0 = pack_bf16x2(x[0], x[1]), w1 = pack_bf16x2(x[2], x[3]);
    uint32_t sbyte;
    const uint32_t codes = quantize4_words(w0, w1, sbyte);
    if (act && n < o.N) {
      const int row_bytes = o.N >> 1;
      uint8_t* dst = o.qcodes + static_cast<size_t>(r) * row_bytes + (n >> 1);
      if (n + 4 <= o.N && (reinterpret_cast<uintptr_t>(dst) & 1) == 0) {
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes);
      } else {
        dst[0] = static_cast<uint8_t>(codes);
        if ((n >> 1) + 1 < row_bytes) dst[1] = static_cast<uint8_t>(codes >> 8);
      }
      if (sub == 0) o.qscales[static_cast<size_t>(r) * ((o.N + 31) >> 5) + (n >> 5)] = static_cast<uint8_t>(sbyte);
    }
  }
}

// kOut: 0 bf16 output, 1 MXFP4 output (g.o.qcodes set), 2 the split + cat
// form (g.o.splitcat set); the bf16 instantiation holds none of the other forms'
// code.
template <int kRowsA, int kOut>
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
  const bool prequant = g.x == nullptr;
  // This CTA's work: tiles t0, t0 + t_step, ... (n_my tiles), k-steps
  // [k0, k0 + nk) of each.  Stage i is k-step k0 + i % nk of tile
  // t0 + (i / nk) * t_step.
  int t0, t_step, n_my, k0, nk;
  if (g.split > 1) {
    const int rank = blockIdx.x % g.split;
    t0 = blockIdx.x / g.split;
    t_step = 0;
    n_my = 1;
    k0 = rank * g.KT / g.split;
    nk = (rank + 1) * g.KT / g.split - k0;
  } else {
    t0 = blockIdx.x;
    t_step = gridDim.x;
    n_my = (g.n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
    k0 = 0;
    nk = g.KT;
  }
  const int n_stages = n_my * nk;
  // Quantizing warps: all of warps 2..9 when each CTA has one tile; else
  // warps 2, 3, 6, 7 only, so that the drain of one tile (warps 4, 5, 8, 9)
  // never waits behind the quantization of the next.
  const bool multi_tile = g.split == 1 && g.n_tiles > static_cast<int>(gridDim.x);
  const int n_qwarps = multi_tile ? 4 : 8;
  bool abort = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // weights: the producer's arrival (+ bytes); activations: one arrival
      // per quantizing warp, or the producer's second arrival (+ bytes)
      mbar_init(&full[s], prequant ? 2 : 1 + n_qwarps);
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
  if (threadIdx.x == 0) {
    griddep_launch_dependents();
    MX_STAMP(0);
  }

  if (warp == 0) {
    // ---- producer: the weight block of each stage (one bulk copy), and in
    // the pre-quantized mode the stage's activation codes and scales.
    // Weights are read once: evict-first keeps L2 for everything else.
    const uint64_t evict_first = policy_evict_first();
    auto w_load = [&](int i, uint8_t* st, uint64_t* bar) {
      const int t = t0 + (i / nk) * t_step, kt = k0 + i % nk;
      bulk_g2s_hint(st, g.w_packed + static_cast<size_t>(t * g.KT + kt) * kWeightBlockBytes, kWeightBlockBytes,
                    bar, evict_first);
    };
    // Activations of the stage's k-step (rows 0..kRowsA-1 of row tile 0):
    // one copy of the blocked form, or codes + scales of the TILED form.
    auto a_load = [&](int i, uint8_t* st, uint64_t* bar) {
      const int kt = k0 + i % nk;
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(C::kALoad + C::kSA));
      if (g.a_blocked) {
        bulk_g2s(st + C::kW, g.a_codes + static_cast<size_t>(kt) * (C::kALoad + C::kSA), C::kALoad + C::kSA, bar);
      } else {
        bulk_g2s(st + C::kW, g.a_codes + (static_cast<size_t>(kt) << 14), C::kALoad, bar);
        bulk_g2s(st + C::kW + C::kA, g.a_scales + (static_cast<size_t>(kt) << 10), C::kSA, bar);
      }
    };
    const int npre = n_stages < C::kStages ? n_stages : C::kStages;
    // Lane i requests the weights of prologue stage i at once.
    if (lane < npre) {
      mbar_arrive_expect_tx(&full[lane], static_cast<uint32_t>(C::kW));
      w_load(lane, smem + lane * C::kStageBytes, &full[lane]);
    }
    if (lane == 0) MX_STAMP(1);
    if (prequant) {
      griddep_wait();   // the activations may come from the kernel before this one
      if (lane < npre) a_load(lane, smem + lane * C::kStageBytes, &full[lane]);
    }
    __syncwarp();
    if (lane == 0) {
      for (int i = npre; i < n_stages; ++i) {
        const int s = i % C::kStages;
        if (!mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, abort)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(C::kW));
        w_load(i, st, &full[s]);
        if (prequant) a_load(i, st, &full[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: one accumulator, one tile at a time
    if (lane == 0) {
      int i = 0;
      for (int tl = 0; tl < n_my && !abort; ++tl) {
        if (!mbar_wait(acc_empty, (tl & 1) ^ 1, abort)) break;
        tc_fence_after();
        for (int j = 0; j < nk; ++j, ++i) {
          const int s = i % C::kStages;
          if (!mbar_wait(&full[s], (i / C::kStages) & 1, abort)) break;
          tc_fence_after();
          if (i == 0) MX_STAMP(3);
          issue_stage_mma<C>(tmem, smem_u32(smem + s * C::kStageBytes), s, j != 0 ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        mma_commit(acc_full);
      }
      MX_STAMP(4);
      // TMEM is freed only after the last drain has read the accumulator.
      mbar_wait(acc_empty, (n_my & 1) ^ 1, abort);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  } else {
    // ---- warps 2..9: activation quantization, then the accumulator drain.
    // x, the bias and the outputs are touched only after the kernel this one
    // depends on has completed.  An L2 prefetch returns no data (L2 is
    // coherent), so the rows a warp quantizes may be requested before that.
    if (!prequant && g.vec_ok != 0 && lane == 0) {
      const int wq = multi_tile ? (warp & 1) + ((warp >> 1) & 2) : warp - 2;
      if (!multi_tile || (warp & 3) >= 2) {
        const int e0 = k0 * 256;
        const int e1 = (k0 + nk) * 256 < g.K ? (k0 + nk) * 256 : g.K;
        const uint32_t bytes = static_cast<uint32_t>(2 * (e1 - e0)) & ~15u;
        for (int r = wq; r < g.M && bytes != 0; r += n_qwarps)
          bulk_prefetch_l2(g.x + static_cast<size_t>(r) * g.ldx + e0, bytes);
      }
    }
    griddep_wait();
    if (threadIdx.x == 64) MX_STAMP(2);
    const int w = multi_tile ? (warp & 1) + ((warp >> 1) & 2) : warp - 2;
    if (!prequant && (!multi_tile || (warp & 3) >= 2)) {
      // Items (stage i, row r) for rows r = w, w + n_qwarps, ... < M, in stage
      // order; kLoadAhead items' x loads are in flight ahead of the one being
      // quantized.  A warp arrives on full[s] once it has written all its
      // rows of the stage (a warp without rows arrives at once), always after
      // the slot was released, so its arrival counts for that stage.
      const int rows_w = g.M > w ? (g.M - 1 - w) / n_qwarps + 1 : 0;
      const int nb = (g.K + 31) >> 5;
      const bool vec_ok = g.vec_ok != 0;
      if (rows_w == 0) {
        for (int i = 0; i < n_stages; ++i) {
          const int s = i % C::kStages;
          if (i >= C::kStages && !mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, abort)) break;
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
        }
      } else {
        const int n_items = n_stages * rows_w;
        uint4 buf[kLoadAhead];
        int li = 0, lq = 0;   // next item to load: stage li, row index lq
        auto load_next = [&]() -> uint4 {
          const int kt = k0 + li % nk;
          const uint4 v = load8_words(g.x, w + n_qwarps * lq, g.M, g.K, g.ldx, kt * 256 + lane * 8, vec_ok);
          if (++lq == rows_w) {
            lq = 0;
            ++li;
          }
          return v;
        };
#pragma unroll
        for (int p = 0; p < kLoadAhead; ++p)
          if (p < n_items) buf[p] = load_next();
        int ci = 0, cq = 0;   // item being quantized
        for (int j0 = 0; j0 < n_items; j0 += kLoadAhead) {
#pragma unroll
          for (int p = 0; p < kLoadAhead; ++p) {
            if (j0 + p >= n_items) break;   // warp-uniform
            const int s = ci % C::kStages;
            if (cq == 0 && ci >= C::kStages) mbar_wait(&empty[s], ((ci / C::kStages) & 1) ^ 1, abort);
            const int r = w + n_qwarps * cq;
            const int kt = k0 + ci % nk;
            uint32_t sbyte;
            const uint32_t packed = quantize8_words(buf[p], sbyte);
            if (j0 + p + kLoadAhead < n_items) buf[p] = load_next();
            uint8_t* a_st = smem + s * C::kStageBytes + C::kW;
            *reinterpret_cast<uint32_t*>(a_st + r * 128 + ((((lane >> 2) ^ (r & 7))) << 4) + ((lane & 3) << 2)) =
                packed;
            if ((lane & 3) == 0) {
              const int b = lane >> 2;   // block of the k-step
              a_st[C::kA + ((b >> 2) << 9) + ((r & 31) << 4) + ((r >> 5) << 2) + (b & 3)] =
                  kt * 8 + b < nb ? static_cast<uint8_t>(sbyte) : static_cast<uint8_t>(0x7F);
            }
            if (++cq == rows_w) {
              // The stage's operands are read by the tensor core (async proxy).
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&full[s]);
              cq = 0;
              ++ci;
            }
          }
        }
      }
    }

    if ((warp & 3) < 2) {
      // ---- drain: warp w% 4 = q reads accumulator rows 32q.., columns 128h..
      // (h = 0 for warps 4, 5; 1 for warps 8, 9).  A whole tile is stored
      // with the bias; a split tile's part goes to this CTA's shared memory.
      const int q = warp & 3;
      const int h = (warp - 2) >> 2;
      const int rl = q * 32 + lane;                 // accumulator row = activation row
      const bool warp_live = q * 32 < g.M;
      const bool live = rl < g.M;
      const uint32_t pbase = smem_u32(smem);
      for (int tl = 0; tl < n_my; ++tl) {
        const int t = t0 + tl * t_step;
        const bool ok = mbar_wait(acc_full, tl & 1, abort);
        tc_fence_after();
        if (threadIdx.x == 128 && tl == n_my - 1) MX_STAMP(5);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          uint32_t r[64];
          if (warp_live) {
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16)
              tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + pass * 64 + c0,
                        *reinterpret_cast<uint32_t(*)[16]>(&r[c0]));
            tmem_wait_ld();
          }
          if (pass == 1) {
            tc_fence_before();
            mbar_arrive(acc_empty);   // the accumulator may be overwritten now
          }
          if (!live) continue;
          if (!ok) {
#pragma unroll
            for (int c = 0; c < 64; ++c) r[c] = 0u;
          }
          if (g.split == 1) {
            const int n0 = t * kTileN + h * 128 + pass * 64;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
              float chunk[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) chunk[c] = __uint_as_float(r[c0 + c]);
              if (kOut == 1)
                store_chunk_q(g.o, rl, n0 + c0, chunk);
              else if (kOut == 2)
                store_chunk_sc(g.o, rl, n0 + c0, chunk);
              else
                store_chunk_bf16(g.o, rl, n0 + c0, chunk);
            }
          } else {
            const int qc0 = (h * 128 + pass * 64) >> 2;
#pragma unroll
            for (int c = 0; c < 16; ++c)
              st_shared_f4(pbase + partial_off(rl, qc0 + c), r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
          }
        }
      }
    }
  }

  if (g.split > 1) {
    // ---- split tile: after every part is in its CTA's shared memory, CTA of
    // rank j sums column chunks [64 j / S, 64 (j + 1) / S) of every live row
    // over the S parts in rank order, adds the bias and stores bf16.  The
    // second barrier keeps every CTA's shared memory alive until all reads
    // of it are done.
    cluster_sync_all();
    if (threadIdx.x == 0) MX_STAMP(6);
    if (warp >= 2) {
      const int S = g.split;
      const int rank = blockIdx.x % S;
      const int q_lo = rank * 64 / S, nq = (rank + 1) * 64 / S - q_lo;
      const uint32_t pbase = smem_u32(smem);
      const int n0 = t0 * kTileN;
      if (kOut == 1) split_sum_store_q(g.o, g.M, S, rank, pbase, n0);
      for (int gi = threadIdx.x - 64; kOut != 1 && gi < g.M * nq; gi += kEpiThreads) {
        const int r = gi / nq, qq = q_lo + gi % nq;
        const uint32_t a = pbase + partial_off(r, qq);
        float4 p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < S) p[k] = ld_shared_cluster_f4(mapa_shared(a, static_cast<uint32_t>(k)));
        float4 acc = p[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) {
          if (k < S) {
            acc.x += p[k].x;
            acc.y += p[k].y;
            acc.z += p[k].z;
            acc.w += p[k].w;
          }
        }
        if (kOut == 2)
          store_quad_sc(g.o, r, n0 + 4 * qq, acc);
        else
          store_quad(g.o, r, n0 + 4 * qq, acc);
      }
    }
    cluster_sync_all();
  }
#ifdef MXFP4_STAMPS
  __syncthreads();   // "done" = the whole CTA has finished (no thread returns early)
#endif
  if (threadIdx.x == 0) MX_STAMP(7);
  if (abort) atomicOr(&g_decode_error, kErrTimeout);
}

// ===================================================================== host
// Per-device, per-kernel host caches; several host threads may fill them
// at once, each writing the same value.
static std::atomic<bool> g_attr_set[64][9];
#ifdef MXFP4_STAMPS
static std::atomic<int> g_stamp_next{0};   // stamp slot of the next launch (in launch order)
#endif
static std::atomic<int> g_max_clusters[64][9][9];   // co-resident clusters of size S (0: not yet queried)

template <int kRowsA, int kOut>
static cudaError_t prepare(const DeviceInfo& dev, int which) {
  using C = Cfg<kRowsA>;
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev.device][which].load(std::memory_order_acquire)) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<kRowsA, kOut>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    g_attr_set[dev.device][which].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

// How many clusters of S CTAs (one per SM) the device holds at once.
template <int kRowsA, int kOut>
static int max_clusters(int S, const DeviceInfo& dev, int which) {
  using C = Cfg<kRowsA>;
  std::atomic<int>& slot = g_max_clusters[dev.device][which][S];
  int cached = slot.load(std::memory_order_acquire);
  if (cached == 0) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<kRowsA, kOut>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached = n > 0 ? n : -1;
    slot.store(cached, std::memory_order_release);
  }
  return cached;
}

template <int kRowsA, int kOut>
static cudaError_t launch_rows(DecodeArgs a, const DeviceInfo& dev, cudaStream_t s, int which) {
  using C = Cfg<kRowsA>;
  cudaError_t e = prepare<kRowsA, kOut>(dev, which);
  if (e != cudaSuccess) return e;
  // Split: with fewer tiles than SMs, S CTAs per tile (a cluster), S as
  // large as the SMs allow (at most 8 and at most one k-step per CTA) with
  // every tile's cluster resident at once; else whole tiles per CTA.
  int split = 1;
  if (a.n_tiles < dev.sm_count) {
    split = dev.sm_count / a.n_tiles;
    if (split > 8) split = 8;
    if (split > a.KT) split = a.KT;
    while (split > 1 && max_clusters<kRowsA, kOut>(split, dev, which) < a.n_tiles) --split;
  }
  a.split = split;
  const int grid = split > 1 ? a.n_tiles * split : (a.n_tiles < dev.sm_count ? a.n_tiles : dev.sm_count);

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(C::kSmem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(split);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<kRowsA, kOut>, a);
}

cudaError_t launch_decode(const DecodeProblem& p, const DeviceInfo& dev, cudaStream_t s) {
  DecodeArgs a{};
  a.x = static_cast<const uint16_t*>(p.x);
  a.ldx = p.ldx;
  a.vec_ok = p.x != nullptr && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 && (p.ldx % 8) == 0;
  a.a_codes = p.a_codes;
  a.a_scales = p.a_scales;
  a.a_blocked = p.a_blocked ? 1 : 0;
  a.w_packed = p.w_packed;
  a.o.out = static_cast<__nv_bfloat16*>(p.out);
  a.o.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.o.ldo = p.ldo;
  a.o.N = p.N;
  a.o.qcodes = p.qcodes;
  a.o.qscales = p.qscales;
  a.o.cat = static_cast<__nv_bfloat16*>(p.cat);
  a.o.split = static_cast<__nv_bfloat16*>(p.split);
  a.o.z = static_cast<const __nv_bfloat16*>(p.z);
  a.o.s1 = p.s1;
  a.o.s2 = p.s2;
  a.o.s3 = p.s3;
  a.o.splitcat = p.splitcat ? 1 : 0;
  a.M = p.M;
  a.K = p.K;
  a.KT = static_cast<int>(padded_k(p.K) / kKTile);
  a.n_tiles = static_cast<int>(ceil_div(p.N, kTileN));
#ifdef MXFP4_STAMPS
  a.stamp_call = g_stamp_next.fetch_add(1) & 0x7FFFFFFF;
#endif
  if (p.qcodes != nullptr) {
    switch (gemm_rows_a(p.M)) {
      case 16: return launch_rows<16, 1>(a, dev, s, 3);
      case 32: return launch_rows<32, 1>(a, dev, s, 4);
      default: return launch_rows<64, 1>(a, dev, s, 5);
    }
  }
  if (p.splitcat) {
    switch (gemm_rows_a(p.M)) {
      case 16: return launch_rows<16, 2>(a, dev, s, 6);
      case 32: return launch_rows<32, 2>(a, dev, s, 7);
      default: return launch_rows<64, 2>(a, dev, s, 8);
    }
  }
  switch (gemm_rows_a(p.M)) {
    case 16: return launch_rows<16, 0>(a, dev, s, 0);
    case 32: return launch_rows<32, 0>(a, dev, s, 1);
    default: return launch_rows<64, 0>(a, dev, s, 2);
  }
}

#ifdef MXFP4_STAMPS
int decode_stamps(unsigned long long* host, int* next_call) {
  *next_call = g_stamp_next.load();
  if (cudaMemcpyFromSymbol(host, g_stamps, sizeof(g_stamps)) != cudaSuccess) return -1;
  return kStampCalls * kStampCtas * kStampPoints;
}
#else
int decode_stamps(unsigned long long*, int*) { return 0; }
#endif

uint32_t decode_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero));
  return v;
}

}  // namespace mx
