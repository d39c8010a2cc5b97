// W4A4 MXFP4 GEMM on the sm_103a block-scaled tensor cores, for M > 64
// (the decode shapes, M <= 64, run in decode.cu).
//
//   out[m][n] = bf16_RNE( sum_k deq(A)[m][k] * deq(W)[n][k] + bias[n] )
//
// the gemm_a4w4 + bias step of sglang PR #39598 (blog analysis, section 2,
// apply_weights).  The weights arrive packed and the activations in the
// library's blocked form (from the quantizer) or the caller's TILED layout,
// so every stage is one or two contiguous 1-D bulk copies: code tiles
// already in the 128-byte-swizzled K-major image, 512-byte scale atoms
// already in the tcgen05.cp source layout.
//
// An output tile is 128 activation rows (the MMA's M) by 256 weight rows
// (its N): a tcgen05.mma.kind::mxf4.block_scale instruction costs about the
// same for any N, so the 256-row weight side does the most work per issued
// instruction.  The (tile, 256-wide k-step) iteration space is split evenly
// over one CTA per SM (stream-K).  Tiles cut by a CTA boundary are published
// as fp32 parts and summed, in CTA order (deterministic), by a fix-up kernel
// launched behind the GEMM.
//
// Roles (320 threads): warp 0 streams stages with bulk copies; warp 1 issues
// tcgen05.cp (scales -> TMEM) and the MMAs into one 128 x 256 fp32 TMEM
// accumulator; warps 2..9 drain it (each 32 rows x 128 columns) with
// tcgen05.ld, release it at once, then add the bias and store bf16 (or
// publish the part).  The tensor pipe bounds the kernel: per 256-wide
// k-step its four MMAs and the scale copies run back to back, so for
// K <= 6144 the activation scales of every k-step stay in TMEM across the
// tiles of one activation row tile (four copies per k-step instead of six).
// With an MXFP4 output (OutView::qcodes set) the epilogue threads quantize
// their 32-column chunks instead of storing bf16, and the fix-up kernel's
// <true> form sums one (row, 32-column block) per thread.  The kernel is
// launched as a programmatic dependent:
// it sets up and requests its first weight stages while the activation
// quantizer before it finishes, and lets the next kernel launch early.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mx {

static __device__ uint32_t g_gemm_error;

struct GemmArgs {
  const uint8_t* a_codes;          // TILED codes, or blocked activations (a_blocked)
  const uint8_t* a_scales;
  int a_blocked;
  const uint8_t* w_packed;         // packed weight blocks
  OutView o;
  int M, KT;
  int n_tiles;                     // ceil(N / 256)
  int total;                       // output tiles x KT
  int grid;
  int rows_a;                      // activation rows per tile that are loaded (128)
  float* partials;                 // 2 slots per CTA, rows_a x 256 floats each
  int whole_tiles;                 // 1: each CTA takes whole tiles (no part is published)
};

// First iteration of CTA c: the balanced stream-K split of the (tile,
// k-step) space, or, with whole tiles, the balanced split of the tiles.
__device__ __forceinline__ int cta_begin(const GemmArgs& g, int c) {
  if (g.whole_tiles) return static_cast<int>((static_cast<long long>(c) * (g.total / g.KT)) / g.grid) * g.KT;
  return sk_begin(c, g.total, g.grid);
}

// One CTA per SM (the ring takes the shared memory), so the full register
// budget of a 320-thread block is available: the epilogue holds a whole
// 128-column accumulator row in registers.
template <int kRowsA>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const GemmArgs g) {
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
  const int it0 = cta_begin(g, cta);
  const int it1 = cta_begin(g, cta + 1);
  bool abort = false;

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
  // touches memory (griddepcontrol.wait), so it may be launched right away;
  // its CTAs take SMs as this kernel's CTAs leave.
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ---- producer.  A stage is one 256-wide k-step of one output tile.
    auto w_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int t = it / KT, kt = it - t * KT;
      const int nt = t % g.n_tiles;
      bulk_g2s(st, g.w_packed + static_cast<size_t>(nt * KT + kt) * kWeightBlockBytes, kWeightBlockBytes, bar);
    };
    auto a_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int t = it / KT, kt = it - t * KT;
      const int mt = t / g.n_tiles;
      if (g.a_blocked) {
        bulk_g2s(st + C::kW, g.a_codes + static_cast<size_t>(mt * KT + kt) * (C::kALoad + C::kSA), C::kALoad + C::kSA,
                 bar);
      } else {
        bulk_g2s(st + C::kW, g.a_codes + (static_cast<size_t>(mt * KT + kt) << 14), C::kALoad, bar);
        bulk_g2s(st + C::kW + C::kA, g.a_scales + (static_cast<size_t>(mt * KT + kt) << 10), 1024, bar);
      }
    };
    auto stage_bytes = [&](int) -> uint32_t { return static_cast<uint32_t>(C::kW + C::kALoad + C::kSA); };
    const int n_iter = it1 - it0;
    const int npre = n_iter < C::kStages ? n_iter : C::kStages;
    // Lane i issues prologue stage i (one copy instruction per lane rather
    // than a serial chain).  Weights are requested before waiting on the
    // activation-producing kernel: the kernel this one follows never writes
    // them (the weight repack ends with an ordinary launch).
    if (lane < npre) {
      uint8_t* st = smem + lane * C::kStageBytes;
      mbar_arrive_expect_tx(&full[lane], stage_bytes(it0 + lane));
      w_load(it0 + lane, st, &full[lane]);
      griddep_wait();
      a_load(it0 + lane, st, &full[lane]);
    }
    __syncwarp();
    if (lane == 0 && npre < n_iter) {
      // The stage's tile and k-step advance one iteration at a time, so no
      // division sits between a stage's release and its copies.  The
      // producer's time per stage is on the kernel's critical path: this
      // measured 0.8% faster than dividing.
      int t = (it0 + npre) / KT, kt = (it0 + npre) - t * KT;
      int mt = t / g.n_tiles, nt = t - mt * g.n_tiles;
      for (int i = npre; i < n_iter; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, abort)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes(it0 + i));
        bulk_g2s(st, g.w_packed + static_cast<size_t>(nt * KT + kt) * kWeightBlockBytes, kWeightBlockBytes, &full[s]);
        const size_t ai = static_cast<size_t>(mt * KT + kt);
        if (g.a_blocked) {
          bulk_g2s(st + C::kW, g.a_codes + ai * (C::kALoad + C::kSA), C::kALoad + C::kSA, &full[s]);
        } else {
          bulk_g2s(st + C::kW, g.a_codes + (ai << 14), C::kALoad, &full[s]);
          bulk_g2s(st + C::kW + C::kA, g.a_scales + (ai << 10), 1024, &full[s]);
        }
        if (++kt == KT) {
          kt = 0;
          if (++nt == g.n_tiles) {
            nt = 0;
            ++mt;
          }
        }
      }
    }
    __syncwarp();   // whole warp reaches the final barrier converged
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: one accumulator, one segment (part of a tile) at a
      // time.  Consecutive tiles of a CTA share their activation rows (tile
      // t = mt * n_tiles + nt), so when every k-step's activation scales fit
      // in TMEM past the accumulator and 16-column weight-scale slots
      // (K <= 6144) they are copied once per activation row tile and k-step
      // and reused: four scale copies per stage instead of six.  (The tensor
      // pipe runs copies and MMAs in issue order, so a row tile's scales
      // overwrite the previous one's only after the MMAs that read them.)
      constexpr uint32_t kSfaRes = C::kSfBase + C::kStages * 16u;
      const bool resident = kSfaRes + 8u * static_cast<uint32_t>(KT) <= C::kTmemCols;
      int cur_mt = -1;
      uint32_t have = 0;   // k-steps whose activation scales of row tile cur_mt are in TMEM
      int i = 0, seg = 0, kt = it0 % KT;
      for (int it = it0; it < it1 && !abort; ++seg) {
        const int len = (KT - kt) < (it1 - it) ? (KT - kt) : (it1 - it);
        const int mt = (it / KT) / g.n_tiles;
        if (mt != cur_mt) {
          cur_mt = mt;
          have = 0;
        }
        for (int j = 0; j < len; ++j, ++i) {
          const int s = i % C::kStages;
          const uint32_t ph = (i / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, abort)) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const int k = kt + j;
          const uint32_t sfa_col = resident ? kSfaRes + 8u * k : C::kSfBase + s * C::kSfSlot;
          const uint32_t sfb_col = resident ? C::kSfBase + 16u * s : sfa_col + C::kSfbOff;
          // the scale copies first: at a segment start they run while the
          // epilogue still drains the previous segment's accumulator
          issue_stage_scales_sfa<C>(tmem, st, sfb_col, sfa_col, !resident || ((have >> k) & 1u) == 0);
          if (resident) have |= 1u << k;
          if (j == 0) {
            if (!mbar_wait(acc_empty, (seg & 1) ^ 1, abort)) break;
            tc_fence_after();
          }
          issue_stage_mmas_sfa<C>(tmem, st, sfb_col, sfa_col, j != 0 ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        mma_commit(acc_full);
        it += len;
        kt = 0;
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: warp w drains accumulator rows 32*(w%4).., columns 128*h..
    griddep_wait();
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int rl = q * 32 + lane;                 // accumulator row = activation row in the tile
    const bool warp_live = q * 32 < kRowsA;       // quarters beyond kRowsA rows hold nothing
    int seg = 0, kt = it0 % KT;
    for (int it = it0; it < it1; ++seg) {
      const int len = (KT - kt) < (it1 - it) ? (KT - kt) : (it1 - it);
      const int t = it / KT;
      const int mt = t / g.n_tiles, nt = t - mt * g.n_tiles;
      const bool ok = mbar_wait(acc_full, seg & 1, abort);
      tc_fence_after();
      const int m = mt * 128 + rl;
      const int n0 = nt * kTileN + h * 128;
      const bool live = warp_live && rl < kRowsA && m < g.M;
      const bool whole = kt == 0 && len == KT;
      const int slot = 2 * cta + (it == it0 ? 0 : 1);
      // All 128 columns of this thread's row are read into registers and the
      // accumulator is released before anything is stored, so the next
      // segment's MMAs do not wait on the stores.  A whole tile is stored
      // (+ bias, bf16); a part of a tile is published as fp32 for the fix-up
      // kernel that follows.
      uint32_t r[128];
      if (warp_live) {
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 16)
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + c0,
                    *reinterpret_cast<uint32_t(*)[16]>(&r[c0]));
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(acc_empty);                     // accumulator free for the next segment
      if (live) {
        if (!ok) {
#pragma unroll
          for (int c = 0; c < 128; ++c) r[c] = 0u;
        }
        if (whole) {
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            float chunk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) chunk[c] = __uint_as_float(r[c0 + c]);
            store_chunk(g.o, m, n0 + c0, chunk);
          }
        } else {
          uint4* P = reinterpret_cast<uint4*>(g.partials + (static_cast<size_t>(slot) * kRowsA + rl) * kTileN + h * 128);
#pragma unroll
          for (int c = 0; c < 32; ++c) __stcg(P + c, make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]));
        }
      }
      it += len;
      kt = 0;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (abort) atomicOr(&g_gemm_error, kErrTimeout);
}

// ================================================================ CTA pairs
// The same GEMM on 256 x 256 output tiles, each computed by a 2-CTA cluster
// with the cta_group::2 MMA: CTA r of the pair holds activation rows
// 128 r .. 128 r + 127 of the tile and weight rows 128 r .. 128 r + 127 (its
// half of the MMA's B operand), plus the scales of all 256 weight rows.  A
// stage is 35 KiB per CTA instead of 51, so the ring holds six stages
// instead of four, and each SM reads 31% fewer operand bytes.  CTA 0 issues
// the scale copies, MMAs and commits for both; CTA 1 tells it when its half
// of a stage has landed (its MMA warp relays its own stage barrier).  Each
// CTA drains its own 128 accumulator rows.  Whole tiles only.
//
// Measured on the prefill shapes it runs at the single-CTA kernel's speed
// (within 0.6% per shape): per SM the pair's k-step costs the tensor pipe what the
// single CTA's does, and both kernels' producers spend most of a stage
// issuing its bulk copies.  So mxfp4_gemm never takes it; it runs only
// behind the diagnostic entry point mxfp4_diag_gemm_pair.
struct CfgPair {
  static constexpr int kWOff = 0;                            // this CTA's 128 weight rows: one code tile
  static constexpr int kSBOff = kTileBytes;                  // scales of the tile's 256 weight rows (4 atoms)
  static constexpr int kAOff = kTileBytes + 4 * kAtomBytes;  // activation codes, 128 rows
  static constexpr int kSAOff = kAOff + kTileBytes;          // activation scale atoms (2)
  static constexpr int kStageBytes = kSAOff + 2 * kAtomBytes;
  static constexpr int kStages = 6;
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kSmem = kRing + 1024 + 512;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSfBase = 256, kSfSlot = 32, kSfbOff = 8;
};
static_assert(CfgPair::kSmem <= kMaxSmem, "pair ring exceeds shared memory");
static_assert(CfgPair::kAOff % 1024 == 0 && CfgPair::kStageBytes % 1024 == 0, "swizzled tiles need 1 KiB alignment");
static_assert(CfgPair::kSfBase + CfgPair::kStages * CfgPair::kSfSlot <= CfgPair::kTmemCols, "scale slots exceed TMEM");

__global__ void __launch_bounds__(kThreads, 1) gemm_pair_kernel(const GemmArgs g) {
  using C = CfgPair;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRing);   // this CTA's half of the stage landed
  uint64_t* pfull = full + C::kStages;                              // (CTA 0) CTA 1's half landed
  uint64_t* empty = pfull + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 1;                               // (CTA 0) both CTAs drained
  uint64_t* done = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int KT = g.KT;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int it0 = cta_begin(g, pair);
  const int it1 = cta_begin(g, pair + 1);
  const int n_iter = it1 - it0;
  const int last_mt = (g.M - 1) >> 7;   // last 128-row activation tile that exists
  bool abort = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&pfull[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * (kEpiThreads / 32));   // one arrival per epilogue warp of either CTA
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers and TMEM exist before any remote arrival or MMA
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ---- producer: this CTA's half of each stage
    auto w_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int t = it / KT, kt = it - t * KT;
      const int nt = t % g.n_tiles;
      const uint8_t* blk = g.w_packed + static_cast<size_t>(nt * KT + kt) * kWeightBlockBytes;
      if (rank == 0) {
        bulk_g2s(st + C::kWOff, blk, kTileBytes, bar);
        bulk_g2s(st + C::kSBOff, blk + 2 * kTileBytes, 4 * kAtomBytes, bar);
      } else {   // the second code tile and the scales are contiguous in the packed block
        bulk_g2s(st + C::kWOff, blk + kTileBytes, kTileBytes + 4 * kAtomBytes, bar);
      }
    };
    auto a_load = [&](int it, uint8_t* st, uint64_t* bar) {
      const int t = it / KT, kt = it - t * KT;
      int mt = 2 * (t / g.n_tiles) + static_cast<int>(rank);
      mt = mt < last_mt ? mt : last_mt;   // rows past M: any existing tile (never stored)
      if (g.a_blocked) {
        bulk_g2s(st + C::kAOff, g.a_codes + static_cast<size_t>(mt * KT + kt) * (kTileBytes + 2 * kAtomBytes),
                 kTileBytes + 2 * kAtomBytes, bar);
      } else {
        bulk_g2s(st + C::kAOff, g.a_codes + (static_cast<size_t>(mt * KT + kt) << 14), kTileBytes, bar);
        bulk_g2s(st + C::kSAOff, g.a_scales + (static_cast<size_t>(mt * KT + kt) << 10), 2 * kAtomBytes, bar);
      }
    };
    const int npre = n_iter < C::kStages ? n_iter : C::kStages;
    if (lane < npre) {
      uint8_t* st = smem + lane * C::kStageBytes;
      mbar_arrive_expect_tx(&full[lane], C::kStageBytes);
      w_load(it0 + lane, st, &full[lane]);
      griddep_wait();
      a_load(it0 + lane, st, &full[lane]);
    }
    __syncwarp();
    if (lane == 0) {
      for (int i = npre; i < n_iter; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait_cluster(&empty[s], ph ^ 1, abort)) break;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        w_load(it0 + i, st, &full[s]);
        a_load(it0 + i, st, &full[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---- MMA issuer for the pair.  Activation scales stay in TMEM across
      // the tiles of one activation row tile when they fit (as in gemm_kernel).
      constexpr uint32_t kSfaRes = C::kSfBase + C::kStages * 16u;
      const bool resident = kSfaRes + 8u * static_cast<uint32_t>(KT) <= C::kTmemCols;
      int cur_mt = -1;
      uint32_t have = 0;
      int i = 0;
      for (int seg = 0; seg * KT < n_iter && !abort; ++seg) {
        const int mt = ((it0 / KT) + seg) / g.n_tiles;
        if (mt != cur_mt) {
          cur_mt = mt;
          have = 0;
        }
        for (int k = 0; k < KT; ++k, ++i) {
          const int s = i % C::kStages;
          const uint32_t ph = (i / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, abort)) break;
          if (!mbar_wait_cluster(&pfull[s], ph, abort)) break;
          tc_fence_after();
          const uint32_t st = smem_u32(smem + s * C::kStageBytes);
          const uint32_t sfa_col = resident ? kSfaRes + 8u * k : C::kSfBase + s * C::kSfSlot;
          const uint32_t sfb_col = resident ? C::kSfBase + 16u * s : sfa_col + C::kSfbOff;
          const uint32_t sfa = tmem + sfa_col, sfb = tmem + sfb_col;
          if (!resident || ((have >> k) & 1u) == 0) {
            tmem_cp_scales_pair(sfa + 0, sdesc_scales(st + C::kSAOff));
            tmem_cp_scales_pair(sfa + 4, sdesc_scales(st + C::kSAOff + kAtomBytes));
          }
          if (resident) have |= 1u << k;
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int q = 0; q < 2; ++q)
              tmem_cp_scales_pair(sfb + a * 8 + q * 4, sdesc_scales(st + C::kSBOff + q * 2 * kAtomBytes + a * kAtomBytes));
          if (k == 0) {
            if (!mbar_wait_cluster(acc_empty, (seg & 1) ^ 1, abort)) break;
            tc_fence_after();
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t id = idesc_mxf4(256, kTileN, (q & 1) * 2, (q & 1) * 2);
            mma_mxf4_pair(tmem, sdesc_sw128(st + C::kAOff + 32 * q), sdesc_sw128(st + C::kWOff + 32 * q), id,
                          sfa + 4 * (q >> 1), sfb + 8 * (q >> 1), (k != 0 || q != 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty[s]);
        }
        mma_commit_pair(acc_full);
      }
      mma_commit_pair(done);   // arrives in both CTAs once every MMA above has completed
    } else if (lane == 0) {
      // ---- CTA 1: pass each landed stage on to CTA 0's issuer
      const uint32_t pf0 = mapa_shared(smem_u32(pfull), 0);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % C::kStages;
        if (!mbar_wait(&full[s], (i / C::kStages) & 1, abort)) break;
        mbar_arrive_cluster_relaxed(pf0 + 8u * static_cast<uint32_t>(s));
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: warp w drains this CTA's accumulator rows 32*(w%4).., columns 128*h..
    griddep_wait();
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int rl = q * 32 + lane;
    const uint32_t ae0 = mapa_shared(smem_u32(acc_empty), 0);
    for (int seg = 0; seg * KT < n_iter; ++seg) {
      const int t = it0 / KT + seg;
      const int mt = 2 * (t / g.n_tiles) + static_cast<int>(rank), nt = t % g.n_tiles;
      const bool ok = mbar_wait_cluster(acc_full, seg & 1, abort);
      tc_fence_after();
      const int m = mt * 128 + rl;
      const int n0 = nt * kTileN + h * 128;
      uint32_t r[128];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 16)
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128 + c0,
                  *reinterpret_cast<uint32_t(*)[16]>(&r[c0]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(ae0);   // this warp's part of the accumulator is free
      if (m < g.M) {
        if (!ok) {
#pragma unroll
          for (int c = 0; c < 128; ++c) r[c] = 0u;
        }
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          float chunk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) chunk[c] = __uint_as_float(r[c0 + c]);
          store_chunk(g.o, m, n0 + c0, chunk);
        }
      }
    }
  }
  // No MMA of the pair is in flight when the TMEM is freed: both CTAs wait
  // for the issuer's last commit.
  if (warp == 1 && lane == 0) {
    bool late = false;
    mbar_wait_cluster(done, 0, late);
    abort = abort || late;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
  if (abort) atomicOr(&g_gemm_error, kErrTimeout);
}

// ===================================================================== fix-up
// Tiles split between CTAs, summed after the GEMM.  Block (x, y) takes
// split tile x, float4 groups [512 y, 512 y + 512) of it (group gi = row
// gi / 64, columns 4 * (gi % 64)..); each group adds the contributors' fp32
// parts in CTA order (deterministic), then the bias, and is stored as bf16.
// Loads of 4 contributors x 2 groups per thread are in flight together.
constexpr int kMaxSplitTiles = kMaxStreamKCtas;
constexpr int kFixupGroups = 512;
struct FixupArgs {
  GemmArgs g;
  int tiles[kMaxSplitTiles];
};

// At most 64 registers per thread, so a waiting fix-up block fits on an SM
// next to a resident GEMM CTA (of the next call).
// kQuant: MXFP4 output (g.o.qcodes set).
template <bool kQuant>
__global__ void __launch_bounds__(256, 4) gemm_fixup_kernel(const __grid_constant__ FixupArgs f) {
  griddep_launch_dependents();
  griddep_wait();                                   // the GEMM's parts are complete and visible
  const GemmArgs& g = f.g;
  const int KT = g.KT;
  const int t = f.tiles[blockIdx.x];
  const int mt = t / g.n_tiles, nt = t - mt * g.n_tiles;
  const int c_lo = sk_owner(t * KT, g.total, g.grid);
  const int c_hi = sk_owner(t * KT + KT - 1, g.total, g.grid);
  const int rows = (g.M - mt * 128) < g.rows_a ? (g.M - mt * 128) : g.rows_a;
  if (kQuant) {
    // MXFP4 output: one (row, 32-column block) per thread, the same sums in
    // the same order (8 float4 groups of the row, contributors in CTA order).
    const int u = blockIdx.y * 256 + threadIdx.x;
    if (u >= rows * (kTileN / 32)) return;
    const int row = u / (kTileN / 32), blk = u % (kTileN / 32);
    const int gq0 = row * (kTileN / 4) + blk * 8;
    float4 acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = c_lo; cc <= c_hi; ++cc) {
      const int sl = 2 * cc + (sk_begin(cc, g.total, g.grid) / KT == t ? 0 : 1);
      const float4* Q = reinterpret_cast<const float4*>(g.partials + static_cast<size_t>(sl) * g.rows_a * kTileN);
      float4 p[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) p[k] = __ldcg(Q + gq0 + k);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc[k].x += p[k].x;
        acc[k].y += p[k].y;
        acc[k].z += p[k].z;
        acc[k].w += p[k].w;
      }
    }
    float v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[4 * k] = acc[k].x;
      v[4 * k + 1] = acc[k].y;
      v[4 * k + 2] = acc[k].z;
      v[4 * k + 3] = acc[k].w;
    }
    store_chunk(g.o, mt * 128 + row, nt * kTileN + 32 * blk, v);
    return;
  }
  const int groups = rows * (kTileN / 4);
  const int g0 = blockIdx.y * kFixupGroups + threadIdx.x;   // this thread: groups g0 and g0 + 256
  if (g0 >= groups) return;
  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  for (int cg = c_lo; cg <= c_hi; cg += 4) {
    float4 p[4][2];
#pragma unroll
    for (int jc = 0; jc < 4; ++jc) {
      const int cc = cg + jc;
      if (cc > c_hi) continue;
      const int sl = 2 * cc + (sk_begin(cc, g.total, g.grid) / KT == t ? 0 : 1);
      const float4* Q = reinterpret_cast<const float4*>(g.partials + static_cast<size_t>(sl) * g.rows_a * kTileN);
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (g0 + 256 * j < groups) p[jc][j] = __ldcg(Q + g0 + 256 * j);
    }
#pragma unroll
    for (int jc = 0; jc < 4; ++jc) {
      if (cg + jc > c_hi) continue;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[j].x += p[jc][j].x;
        acc[j].y += p[jc][j].y;
        acc[j].z += p[jc][j].z;
        acc[j].w += p[jc][j].w;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int gi = g0 + 256 * j;
    if (gi < groups) store_quad_any(g.o, mt * 128 + gi / (kTileN / 4), nt * kTileN + 4 * (gi % (kTileN / 4)), acc[j]);
  }
}

// ===================================================================== host
static std::atomic<bool> g_attr_set[64];   // kernel attribute set on this device
static std::atomic<int> g_pairs[64];       // co-resident CTA pairs of gemm_pair_kernel (0: not yet known)

// How many CTA pairs of gemm_pair_kernel the device holds at once (its
// shared-memory attribute set first), or -1 if that cannot be determined.
static int resident_pairs(const DeviceInfo& dev) {
  int n = g_pairs[dev.device].load(std::memory_order_acquire);
  if (n != 0) return n;
  if (cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgPair::kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    n = -1;
  } else {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = CfgPair::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = -1;
    }
  }
  g_pairs[dev.device].store(n, std::memory_order_release);
  return n;
}

// Idle share of the last wave when `units` of work go to `slots` workers.
static double last_wave_idle(int64_t units, int slots) {
  const double waves = static_cast<double>(units) / slots;
  return (static_cast<double>(ceil_div(units, static_cast<int64_t>(slots))) - waves) / waves;
}

int gemm_pair_count(int M, int N, const DeviceInfo& dev) {
  if (M <= kDecodeMaxM || dev.device < 0 || dev.device >= 64) return 0;
  const int64_t n_mt = ceil_div(M, 128);
  const int64_t tiles2 = ceil_div(M, 256) * ceil_div(N, kTileN);
  int pairs = resident_pairs(dev);
  const int grid = gemm_grid(dev);
  if (pairs > grid / 2) pairs = grid / 2;
  if (pairs <= 0) return 0;
  if (pairs > tiles2) pairs = static_cast<int>(tiles2);
  return (n_mt % 2 == 0 || n_mt >= 16) && last_wave_idle(tiles2, pairs) < 0.08 ? pairs : 0;
}


size_t gemm_streamk_workspace_bytes(int M, int N, int K, int grid) {
  (void)N;
  (void)K;
  if (M <= kDecodeMaxM) return 0;   // the decode kernel sums split tiles in shared memory
  return static_cast<size_t>(2) * grid * gemm_rows_a(M) * kTileN * sizeof(float);
}


int gemm_grid(const DeviceInfo& dev) { return dev.sm_count < kMaxStreamKCtas ? dev.sm_count : kMaxStreamKCtas; }

cudaError_t launch_gemm(const GemmProblem& p, const DeviceInfo& dev, cudaStream_t s) {
  GemmArgs a{};
  const int64_t Kp = padded_k(p.K);
  a.a_codes = p.a_codes;
  a.a_scales = p.a_scales;
  a.a_blocked = p.a_blocked ? 1 : 0;
  a.w_packed = p.w_packed;
  a.o.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.o.out = static_cast<__nv_bfloat16*>(p.out);
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
  a.KT = static_cast<int>(Kp / kKTile);
  a.n_tiles = static_cast<int>(ceil_div(p.N, kTileN));
  const int64_t tiles = ceil_div(p.M, 128) * static_cast<int64_t>(a.n_tiles);
  a.total = static_cast<int>(tiles * a.KT);
  int grid = gemm_grid(dev);
  if (grid > a.total) grid = a.total;
  a.grid = grid;
  a.rows_a = gemm_rows_a(p.M);
  a.partials = static_cast<float*>(p.workspace);
  // Whole tiles per CTA when the last wave's idle share is below 8% of the
  // work: the tiles cut by CTA boundaries then cost more (their fp32 parts
  // written and read back, and the fix-up launch) than the idle SMs do
  // (measured: 3% and 8% against 50%, the latter slower at 2.1 waves).
  a.whole_tiles = tiles >= grid && last_wave_idle(tiles, grid) < 0.08 ? 1 : 0;
  if (a.rows_a != 128) return cudaErrorInvalidValue;   // M <= 64 runs in decode.cu
  using C = Cfg<128>;
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (p.cta_pairs) {
    // the CTA-pair kernel on 256-row tiles, whole tiles per pair, or nothing
    const int pairs = gemm_pair_count(p.M, p.N, dev);
    if (pairs <= 0) return cudaErrorNotSupported;
    GemmArgs b = a;
    b.total = static_cast<int>(ceil_div(p.M, 256) * a.n_tiles * a.KT);
    b.grid = pairs;
    b.whole_tiles = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = CfgPair::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, b);
  }
  if (!g_attr_set[dev.device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    g_attr_set[dev.device].store(true, std::memory_order_release);
  }
  cudaError_t e = launch_pdl(gemm_kernel<128>, a.grid, kThreads, C::kSmem, s, a);
  if (e != cudaSuccess) return e;
  // Tiles that a CTA boundary cuts are summed by the fix-up kernel.
  FixupArgs f;
  f.g = a;
  int n_split = 0, prev = -1;
  for (int c = 1; c < grid && !a.whole_tiles; ++c) {
    const int b = static_cast<int>((static_cast<long long>(c) * a.total) / grid);
    if (b % a.KT == 0) continue;
    const int t = b / a.KT;
    if (t != prev) f.tiles[n_split++] = t;
    prev = t;
  }
  if (n_split == 0) return cudaSuccess;
  const int chunks = static_cast<int>(ceil_div(static_cast<int64_t>(a.rows_a) * (kTileN / 4), kFixupGroups));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(n_split), static_cast<unsigned>(chunks), 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.qcodes != nullptr ? cudaLaunchKernelEx(&cfg, gemm_fixup_kernel<true>, f)
                             : cudaLaunchKernelEx(&cfg, gemm_fixup_kernel<false>, f);
}

uint32_t gemm_read_clear_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
  return v;
}

}  // namespace mx
