/*
 * mxfp4_diag.h — diagnostic entry points of the GB300 MXFP4 library.
 *
 * These calls measure the hardware the GEMM kernels run on; they compute
 * nothing of the MXFP4 linear and are not part of its path.  The paper pages
 * have no counterpart: they quote no kernel-level rates (the speed tests of
 * sglang PR #39598 "[AMD] Add opt-in AITER ASM FP4 GEMM for Quark dense
 * linear" are left as a TODO), so the dense FP4 tensor-core rate the GEMM's
 * roofline is quoted against is measured here.
 *
 * Conventions as in mxfp4.h: device pointers are the caller's, every call is
 * asynchronous on `stream` (a cudaStream_t), argument checks return a status
 * before any launch.
 */
#ifndef MXFP4_GB300_DIAG_H
#define MXFP4_GB300_DIAG_H

#include "mxfp4.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest number of measuring units (CTAs, or CTA pairs) one
 * mxfp4_diag_tensor_rate launch reports: the size of its ns_dev buffer. */
MXFP4_API int mxfp4_diag_max_units(void);

/* Tensor-pipe issue rate of one of mxfp4_diag_tensor_rate_variants()
 * instruction mixes, on every SM at once.
 *
 * mxfp4_diag_tensor_rate_info(variant, info) fills info[0..6] with the mix:
 * pair (1: cta_group::2 over a 2-CTA cluster, M = 256; 0: one CTA, M = 128),
 * kind (0: kind::mxf4.block_scale.scale_vec::2X, E2M1 x E2M1 with UE8M0
 * scales, K = 64; 1: kind::f16, bf16 x bf16, K = 16; 2: the kind 0 product
 * issued as kind::mxf4nvf4.block_scale.scale_vec::2X), MMAs per step, scale
 * copies per step, copy form (0: tcgen05.cp.32x128b.warpx4, 1:
 * tcgen05.cp.128x256b), issuing threads per CTA (1, or 2 with separate
 * accumulators of N <= 128 columns each), commit placement (0: the step's
 * groups of four MMAs each after its share of the copies, one commit per
 * step; 1: all the step's copies first, then each group's MMAs followed by
 * a commit of its own; 2: as 0, with each step's commit issued after the
 * next step's copies, just before its MMAs).
 *
 * Each unit (one CTA per SM, or one 2-CTA cluster) issues `steps` steps back
 * to back after 16 untimed ones: the copies and the MMAs of shape
 * M x mma_n x K into the issuer's accumulator, in groups of four MMAs each
 * after its share of the step's copies (one group per 256-wide k-step of
 * the GEMMs), each step committed to an mbarrier, with a wait on the commit of the step `depth` back before the
 * next step is issued (depth 4: the round trip of a 4-stage pipeline ring;
 * depth 32: nearly free issue).  Operands are zero bytes.
 *
 * ns_dev: device buffer of mxfp4_diag_max_units() uint64; unit u's elapsed
 * nanoseconds for the timed steps (%globaltimer; the slower issuer of a
 * two-issuer CTA) land in ns_dev[u], or 0 if a bounded wait gave up.  *units
 * (host) receives the number of units launched.  Arguments: mma_n a multiple
 * of 16 in [16, 256] ([64, 256] for a pair, at most 128 with two issuers),
 * 1 <= steps <= 10^6, 1 <= depth <= 32 (2 <= depth for placement 2); otherwise
 * MXFP4_ERR_INVALID_ARG. */
MXFP4_API int mxfp4_diag_tensor_rate_variants(void);
MXFP4_API mxfp4_status mxfp4_diag_tensor_rate_info(int variant, int* info);
MXFP4_API mxfp4_status mxfp4_diag_tensor_rate(int variant, int mma_n, int steps, int depth,
                                              unsigned long long* ns_dev, int* units, void* stream);

/* One 2-CTA cluster whose CTAs each take 32 TMEM columns with
 * tcgen05.alloc.cta_group::2 (one warp per CTA, as that form requires) and
 * free them again.  addr_dev (device, 2 uint32) receives each CTA's column
 * address with its cluster rank in bits 30..31: equal addresses show that
 * the pair allocated together, which the pair forms of
 * mxfp4_diag_tensor_rate rely on. */
MXFP4_API mxfp4_status mxfp4_diag_pair_alloc_probe(uint32_t* addr_dev, void* stream);

/* Failure-path test hook: sets, for the mxfp4_rmsnorm_quant_act calls that
 * follow in this process, the bound (in SM clock cycles) of its bulk-copy
 * kernel's waits on the row copies; 0 restores the default of about one
 * second.  With a bound far below a copy's latency the wait runs out: the
 * kernel records the timeout (reported by mxfp4_get_device_error as
 * MXFP4_ERR_TIMEOUT), lets every copy it issued land under the full bound,
 * and exits without writing the rows it did not finish.  A test uses this
 * to exercise the bounded-wait path without a fault.  Returns
 * MXFP4_ERR_INVALID_ARG for a negative bound. */
MXFP4_API mxfp4_status mxfp4_diag_set_wait_cycles(long long cycles);

/* Per-call timeline of the decode GEMM kernel (the M <= 64 path of
 * mxfp4_gemm), available only in the library's timeline build (compiled with
 * -DMXFP4_STAMPS; build(variant="timeline")); the default build returns
 * MXFP4_ERR_INVALID_ARG.  Copies to `host` (at least 64*256*8 uint64) the
 * %globaltimer stamps, in ns, of the last 64 decode launches: element
 * [call % 64][cta][point] with points 0 CTA start (after set-up), 1 first
 * weight stages requested, 2 dependency wait passed, 3 first stage's operands
 * complete (MMA thread), 4 last MMAs issued, 5 accumulator complete (drain),
 * 6 split tile: parts visible across the cluster, 7 CTA done.  Point 0
 * carries the launch's sequence number (modulo 2^16) in its top 16 bits and
 * the time in the low 48, so rows left by an older launch in the same slot
 * can be discarded.  *next_call receives the number of decode launches so
 * far (the sequence number of the next one).  Synchronous; stamps of
 * launches still running are partial. */
MXFP4_API mxfp4_status mxfp4_diag_decode_timeline(unsigned long long* host, size_t host_bytes, int* next_call);

/* mxfp4_gemm run on the CTA-pair kernel: 256 x 256 output tiles, each
 * computed by a 2-CTA cluster with tcgen05 cta_group::2 MMAs (each CTA holds
 * 128 activation rows and 128 of the tile's 256 weight rows; six 35 KiB
 * pipeline stages per CTA instead of four of 51 KiB), whole tiles per pair.
 *
 * Same operation, arguments, layouts, workspace and results as mxfp4_gemm
 * with a bf16 output (sglang PR #39598 "[AMD] Add opt-in AITER ASM FP4 GEMM
 * for Quark dense linear", blog analysis section 2, apply_weights: the
 * per-1x32 activation quantization, the W4A4 GEMM with fp32 accumulation,
 * the bias).  It applies where M > 64, the 128-row activation tiles pair up
 * (an even count, or at least 16) and the last wave of 256 x 256 tiles over
 * the device's co-resident CTA pairs is at most 8% idle; elsewhere it
 * returns MXFP4_ERR_UNSUPPORTED_SHAPE before any launch.  mxfp4_gemm never
 * takes this kernel: on the prefill shapes it measured at the single-CTA
 * kernel's speed, not faster (per SM a pair's k-step costs the tensor pipe
 * what a single CTA's does).  It is here so that the comparison can be
 * repeated (python bench.py --prefill-pairs). */
MXFP4_API mxfp4_status mxfp4_diag_gemm_pair(const void* a_bf16_dev, int lda, const uint8_t* a_codes_dev,
                                            const uint8_t* a_scales_dev, mxfp4_layout a_layout,
                                            const void* w_packed_dev, const void* bias_dev, void* out_dev, int ldo,
                                            int M, int N, int K, void* workspace_dev, size_t workspace_bytes,
                                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_DIAG_H */
