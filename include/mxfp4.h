/*
 * mxfp4.h — C ABI of the GB300 (sm_103a) MXFP4 block-scaled dense linear.
 *
 * The library implements the hot path of the MXFP4 dense linear described in
 * sglang PR #39598 "[AMD] Add opt-in AITER ASM FP4 GEMM for Quark dense
 * linear" (and its blog analysis, section 2, the diff of
 * quark_w4a4_mxfp4.py) and the A16WFP4 absorbed BMM of sglang PR #34317
 * "[AMD] [GLM5] use tuned MXFP4 kernels for MLA absorbed BMM".
 *
 * Formats.  An MXFP4 matrix of R rows and K elements (K even) is
 *   - codes:  E2M1 4-bit values, two per byte, element 2j in the low nibble
 *             of byte j, row-major [R][K/2];
 *   - scales: E8M0 bytes (value 2^(e-127), 0xFF = NaN), one per 32
 *             consecutive elements of a row, row-major [R][ceil(K/32)]
 *             (shapes of the pages' per_1x32_f4_quant fake implementation).
 *
 * The TILED layout (MXFP4_LAYOUT_TILED) is this library's repacked form,
 * the layout the tcgen05 block-scaled MMA consumes: rows padded to
 * Rp = ceil(R/128)*128 and elements to Kp = ceil(K/256)*256;
 *   codes region (Rp*Kp/2 bytes): 16 KiB tiles of 128 rows x 128 bytes,
 *     tile (rt,kt) at ((rt*Kp/256)+kt)*16384, byte j of tile row i at
 *     i*128 + ((j/16) ^ (i%8))*16 + j%16 (128-byte swizzle);
 *   scales region (Rp*Kp/32 bytes): 512-byte atoms of 128 rows x 4 scales,
 *     atom (rt,g) at ((rt*Kp/128)+g)*512, scale of atom row i, block b at
 *     16*(i%32) + 4*(i/32) + b%4.
 *   Padding codes are 0 and padding scales 0x7F (E8M0 1.0; the pages pad
 *   with 1.0 because 0xFF is NaN).
 *
 * Packed WEIGHTS use the same tiles and atoms grouped by pairs of row tiles
 * (one bulk copy feeds one MMA stage): rows padded to Np = ceil(N/256)*256;
 * for each pair p (rows 256p..256p+255) and k-tile kt, one 34816-byte block at
 * (p*Kp/256 + kt)*34816 = [code tile of rows 256p.. | code tile of rows
 * 256p+128.. | atoms (block groups 0, 1) of the first 128 rows | atoms of the
 * second 128 rows], 16384 + 16384 + 1024 + 1024 bytes.  A batch of weight
 * matrices is stored back to back.
 *
 * Conventions.
 *   - Pointers named *_dev are device pointers; the caller owns all memory.
 *     Except for the workspace the caller passes, the library allocates
 *     nothing and frees nothing.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Every call is
 *     asynchronous and stream-ordered; argument checks run on the host before
 *     any launch and return their status synchronously.
 *   - Data pointers must be 16-byte aligned (MXFP4_ERR_MISALIGNED).
 *   - No call falls back to another implementation: a shape the kernels do
 *     not support returns MXFP4_ERR_UNSUPPORTED_SHAPE.
 *   - Device-side waits are bounded; a wait that gives up records an error
 *     word that mxfp4_get_device_error() returns as MXFP4_ERR_TIMEOUT.
 */
#ifndef MXFP4_GB300_H
#define MXFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MXFP4_API __attribute__((visibility("default")))
#else
#define MXFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXFP4_OK = 0,
    MXFP4_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, bad enum  */
    MXFP4_ERR_UNSUPPORTED_SHAPE = 2,  /* e.g. odd K, leading dimension too small    */
    MXFP4_ERR_MISALIGNED = 3,         /* pointer or leading dimension not 16-B aligned */
    MXFP4_ERR_WORKSPACE = 4,          /* workspace missing or smaller than required */
    MXFP4_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed       */
    MXFP4_ERR_TIMEOUT = 6,            /* a device-side wait gave up                 */
    MXFP4_ERR_NO_DEVICE = 7           /* no usable sm_103 device is current         */
} mxfp4_status;

typedef enum {
    MXFP4_LAYOUT_ROWMAJOR = 0,  /* codes [R][K/2], scales [R][ceil(K/32)] */
    MXFP4_LAYOUT_TILED = 1      /* the tcgen05 tile layout described above */
} mxfp4_layout;

typedef enum {
    MXFP4_OUT_BMN = 0,  /* out[b][m][n]  (K-up projection)                    */
    MXFP4_OUT_MBN = 1   /* out[m][b][n]  (V-up projection, batch-major write) */
} mxfp4_bmm_out_layout;

/* Version of this ABI (increments on incompatible change; 3: the diagnostic
 * mxfp4_diag_tensor_rate_info of mxfp4_diag.h fills seven ints, not six). */
MXFP4_API int mxfp4_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
MXFP4_API const char* mxfp4_status_string(mxfp4_status status);

/*
 * Bytes of the packed weight buffer for `batch` matrices of N rows x K
 * elements: batch * (Np*Kp/2 + Np*Kp/32) with Np = ceil(N/256)*256.  Returns
 * 0 when an argument is not positive or K is odd.
 */
MXFP4_API size_t mxfp4_packed_weight_bytes(int batch, int N, int K);

/*
 * One-time repack of FP4 weights into the packed weight layout — the counterpart of
 * the pages' process_weights_after_loading step, which swizzles the E8M0
 * weight scales into AITER's tile order and preshuffles the FP4 weights
 * (PR #39598 blog analysis, section 2: _swizzle_asm_fp4_scale,
 * shuffle_weight).  Unlike the pages' gate (rows % 32, scale cols % 8,
 * N > 128) every shape is accepted: rows and K are padded instead.
 *
 *   w_codes_dev   [batch][N][K/2] uint8, row-major, contiguous
 *   w_scales_dev  [batch][N][ceil(K/32)] uint8, row-major, contiguous
 *   packed_dev    mxfp4_packed_weight_bytes(batch, N, K) bytes (output)
 * Deterministic and idempotent.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE
 * (odd K), MISALIGNED, CUDA.
 */
MXFP4_API mxfp4_status mxfp4_pack_weights(const uint8_t* w_codes_dev, const uint8_t* w_scales_dev,
                                int batch, int N, int K, void* packed_dev, void* stream);

/*
 * Orders the GEMM and BMM calls issued next on `stream` after every write to
 * packed weights already issued on it: one empty, ordinary kernel launch.
 * Needed only when a packed weight buffer was written by something other
 * than mxfp4_pack_weights (for example a device-to-device copy refreshing
 * it) and the next kernel on the stream is a GEMM or BMM of this library,
 * which would otherwise start reading the weights before that write has
 * finished (see the weight-update contract of mxfp4_gemm).  No counterpart
 * on the pages, whose weights are written once at load time.
 * Errors: NO_DEVICE, CUDA.
 */
MXFP4_API mxfp4_status mxfp4_weights_updated(void* stream);

/* Bytes of the activation codes / scales buffers for M rows x K elements. */
MXFP4_API size_t mxfp4_act_code_bytes(int M, int K, mxfp4_layout layout);
MXFP4_API size_t mxfp4_act_scale_bytes(int M, int K, mxfp4_layout layout);

/*
 * Per-1x32 MXFP4 quantization of bf16 activations — the pages'
 * per_1x32_f4_quant (PR #39598 blog analysis, section 2,
 * _aiter_per_1x32_f4_quant and its fake implementation for shapes).
 * For each block of 32 elements of a row: amax = max|x|; scale byte =
 * max(biased_exponent(amax) - 2, 0), i.e. the OCP MX exponent
 * floor(log2 amax) - 2 clamped to E8M0; each element is divided by the scale
 * and rounded to the nearest E2M1 value, ties to even, saturating at +-6,
 * keeping the input's sign bit (so -0 encodes as 0x8).  A block holding
 * Inf/NaN gets scale 0xFF and codes 0.  No flush of subnormal inputs.
 *
 *   x_dev       bf16 [M][ldx], ldx >= K (elements)
 *   codes_dev   mxfp4_act_code_bytes(M, K, layout) bytes (output)
 *   scales_dev  mxfp4_act_scale_bytes(M, K, layout) bytes (output)
 * K must be even.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
MXFP4_API mxfp4_status mxfp4_quant_act(const void* x_dev, int M, int K, int ldx,
                             uint8_t* codes_dev, uint8_t* scales_dev,
                             mxfp4_layout layout, void* stream);

/*
 * Fused RMSNorm -> per-1x32 MXFP4 activation producer: the upstream
 * normalization emits the GEMM's quantized input directly.  The pages' layer
 * code accepts such a pre-quantized (codes, scales) tuple and names a fused
 * RMSNorm as one source of it (PR #39598 blog analysis, section 2,
 * apply_weights).  The pages do not print the
 * normalization; it is RMSNorm (Zhang and Sennrich, 2019) with eps inside
 * the root, applied row by row:
 *   h = x                      (residual_dev == NULL), or
 *   h = bf16_RNE(x + residual) (then written back into residual_dev);
 *   y = bf16_RNE( h / sqrt(mean_k(h^2) + eps) * gamma )
 * and y is quantized exactly as mxfp4_quant_act quantizes a bf16 input, so
 * the result equals RMSNorm-to-bf16 followed by mxfp4_quant_act (up to the
 * fp32 evaluation of y: squares and sums in fp32, 1/sqrt by the hardware
 * reciprocal square root; y is within 1 bf16 ulp of the exact value).
 *
 *   x_dev         bf16 [M][ldx], ldx >= K
 *   residual_dev  bf16 [M][ldr], ldr >= K, read and overwritten; or NULL
 *   gamma_dev     bf16 [K]
 *   eps           added to the mean square (>= 0)
 *   codes_dev     mxfp4_act_code_bytes(M, K, layout) bytes (output)
 *   scales_dev    mxfp4_act_scale_bytes(M, K, layout) bytes (output)
 *   y_dev         bf16 [M][ldy], ldy >= K: the bf16 y that was quantized
 *                 (output); or NULL
 * K must be even.  y, codes and scales must not overlap the inputs.  Rows
 * whose mean square leaves the fp32 range (RMS above about 2^63 or below
 * about 2^-63) are outside the supported range.  Launched as a programmatic
 * dependent of the previous kernel on the stream, like mxfp4_quant_act.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
MXFP4_API mxfp4_status mxfp4_rmsnorm_quant_act(const void* x_dev, int ldx, void* residual_dev, int ldr,
                                               const void* gamma_dev, float eps, int M, int K,
                                               uint8_t* codes_dev, uint8_t* scales_dev, mxfp4_layout layout,
                                               void* y_dev, int ldy, void* stream);

/*
 * Workspace bytes mxfp4_gemm needs for this problem (any input form): room
 * for the quantized or re-laid-out activations and, for M > 64, the fp32
 * partial sums of output tiles split between thread blocks.  Its contents
 * need no initialization.
 */
MXFP4_API size_t mxfp4_gemm_workspace_bytes(int M, int N, int K);

/*
 * W4A4 MXFP4 GEMM with fused bias — the pages' gemm_a4w4 followed by
 * `y + bias` (PR #39598 blog analysis, section 2, apply_weights):
 *   out[m][n] = bf16_RNE( sum_k deq(A)[m][k] * deq(W)[n][k] + bias[n] )
 * with deq(c, s) = e2m1(c) * 2^(s-127), fp32 accumulation on the tcgen05
 * block-scaled tensor cores, one rounding to bf16.
 *
 * Activation input, exactly one of:
 *   a_bf16_dev != NULL: bf16 [M][lda] (lda >= K), quantized inside the call
 *                       (the pages' apply_weights path); a_codes/a_scales NULL;
 *   a_bf16_dev == NULL: pre-quantized codes/scales in `a_layout` (the pages'
 *                       (x_fp4, x_scales) tuple input); ROWMAJOR scales are
 *                       re-laid out inside the call.
 *   w_packed_dev   output of mxfp4_pack_weights(batch = 1, N, K)
 *   bias_dev       bf16 [N] or NULL
 *   out_dev        bf16 [M][ldo], ldo >= N
 *   workspace_dev  >= mxfp4_gemm_workspace_bytes(M, N, K) bytes of device
 *                  scratch owned by the caller, clobbered by every call (no
 *                  initialization needed).  One workspace may serve calls of
 *                  any shape; calls sharing one must be ordered on the GPU.
 * For M <= 8 with a bf16 input the whole call is one kernel launch (each
 * thread block quantizes the activations of its own k-range); for
 * 8 < M <= 64 the activation quantizer runs first.
 * Weight-update contract: the GEMM kernel is a programmatic dependent launch
 * that starts streaming the packed weights before the previous kernel in
 * the stream has finished (only its activation, bias and output accesses
 * wait for it).  So the packed weights must not be written by the kernel
 * launched immediately before the call.  mxfp4_pack_weights keeps this true
 * by itself; after writing a packed buffer any other way (a device copy, a
 * foreign kernel), call mxfp4_weights_updated on the stream before the first
 * GEMM or BMM that reads it.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, WORKSPACE, CUDA.
 */
MXFP4_API mxfp4_status mxfp4_gemm(const void* a_bf16_dev, int lda,
                        const uint8_t* a_codes_dev, const uint8_t* a_scales_dev,
                        mxfp4_layout a_layout,
                        const void* w_packed_dev, const void* bias_dev,
                        void* out_dev, int ldo, int M, int N, int K,
                        void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * The same GEMM with an MXFP4 output epilogue: the result, computed and
 * rounded to bf16 exactly as mxfp4_gemm computes it, is quantized per 1x32
 * along N by the rule of mxfp4_quant_act, for the next layer to take as its
 * pre-quantized input.  The pages list a fused MXFP4 output epilogue among
 * the companion changes of their test stack ("[AMD] Add opt-in AITER ASM
 * FP4 GEMM for Quark dense linear", Setup & Environment, companion PR
 * #39912) without printing it; the plainest reading is taken: the bytes
 * equal mxfp4_gemm's bf16 output passed through mxfp4_quant_act (ROWMAJOR).
 *
 *   out_codes_dev   [M][N/2] uint8, row-major (output)
 *   out_scales_dev  [M][ceil(N/32)] uint8, row-major (output)
 * The activation, weight, bias and workspace arguments are mxfp4_gemm's
 * (mxfp4_gemm_workspace_bytes sizes the workspace).  N must be even.  No
 * alignment is required of the outputs (16-byte aligned rows store faster).
 * Errors: those of mxfp4_gemm.
 */
MXFP4_API mxfp4_status mxfp4_gemm_mxfp4_out(const void* a_bf16_dev, int lda,
                                            const uint8_t* a_codes_dev, const uint8_t* a_scales_dev,
                                            mxfp4_layout a_layout, const void* w_packed_dev,
                                            const void* bias_dev, uint8_t* out_codes_dev,
                                            uint8_t* out_scales_dev, int M, int N, int K,
                                            void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * The same GEMM with the split + cat fused epilogue.  The pages name it only:
 * a 5-tuple activation input requests the Triton-only fused "split + cat"
 * epilogue (fused_gemm_afp4wfp4_split_cat), which their ASM path rejects
 * (sglang PR #39598 blog analysis, section 2: _asm_fp4_prequantized_input,
 * the fused_gemm_afp4wfp4_split_cat import; PR #39598 Motivation,
 * "Limitation").  The plainest reading of the name is taken: the GEMM's
 * bf16 result (+ bias), computed and rounded exactly as mxfp4_gemm computes
 * it, is viewed as H = N / (s1 + s2) groups of s1 + s2 columns; the first s1
 * columns of group h are concatenated with the caller's z[m][h] (s3 values)
 * into out_cat, the other s2 go to out_split:
 *   out_cat[m][h][j]        = y[m][h (s1 + s2) + j]          j < s1
 *   out_cat[m][h][s1 + j]   = z[m][h][j]                     j < s3
 *   out_split[m][h][j]      = y[m][h (s1 + s2) + s1 + j]     j < s2
 * (the multi-head key/value projection pattern: per head, a part joined with
 * a separately computed part and a part kept apart).
 *
 *   z_dev          bf16 [M][H][s3], contiguous (ignored when s3 == 0)
 *   out_cat_dev    bf16 [M][H][s1 + s3], contiguous (ignored when s1 + s3 == 0)
 *   out_split_dev  bf16 [M][H][s2], contiguous (ignored when s2 == 0)
 * The activation, weight, bias and workspace arguments are mxfp4_gemm's
 * (mxfp4_gemm_workspace_bytes sizes the workspace).  s1, s2, s3 >= 0,
 * s1 + s2 > 0 (INVALID_ARG); s1, s2, s3 multiples of 8 and N a multiple of
 * s1 + s2 (UNSUPPORTED_SHAPE); the three tensors 16-byte aligned
 * (MISALIGNED).  Other errors: those of mxfp4_gemm.
 */
MXFP4_API mxfp4_status mxfp4_gemm_split_cat(const void* a_bf16_dev, int lda,
                                            const uint8_t* a_codes_dev, const uint8_t* a_scales_dev,
                                            mxfp4_layout a_layout, const void* w_packed_dev,
                                            const void* bias_dev, int M, int N, int K, int s1, int s2,
                                            const void* z_dev, int s3, void* out_cat_dev, void* out_split_dev,
                                            void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * A16WFP4 batched matmul for the MLA absorbed K-up / V-up projections
 * (PR #34317, Modifications): bf16 activations against FP4 weights with E8M0
 * scales, no activation quantization:
 *   r[b][m][n] = bf16_RNE( sum_k x[b][m][k] * deq(W_b)[n][k] ), fp32 accumulation
 *   out_layout BMN: out[b][m][n] = r;  MBN: out[m][b][n] = r (V-up written
 *   batch-major directly, no separate transpose).
 *
 *   x_dev         bf16 [B][M][K], contiguous
 *   w_packed_dev  output of mxfp4_pack_weights(B, N, K)
 *   out_dev       bf16, B*M*N elements in out_layout order
 * Weight-update contract: as for mxfp4_gemm (the weight tile is read and
 * dequantized before the previous kernel in the stream has finished).
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, CUDA.
 */
MXFP4_API mxfp4_status a16wfp4_bmm(const void* x_dev, const void* w_packed_dev, void* out_dev,
                         int B, int M, int N, int K, mxfp4_bmm_out_layout out_layout,
                         void* stream);

/*
 * mxfp4_gemm without a workspace argument, for callers that cannot allocate
 * device memory where they run the layer: code inside CUDA stream capture,
 * serving loops that must not take cudaMalloc's implicit synchronisation,
 * and hosts whose device memory belongs to an allocator this library cannot
 * call.  (The pages have no counterpart; this entry point is an addition.)
 *
 * Same operation and arguments as mxfp4_gemm with a bf16 activation input;
 * the scratch comes from one fixed device array inside the library, of
 * mxfp4_gemm_noalloc_max_scratch_bytes() bytes (48 MiB).  The array is
 * reserved on every device where the library's module is loaded (with eager
 * module loading, every device the process initialises, whether or not this
 * entry point is ever called) and held until the process exits.  A problem whose
 * mxfp4_gemm_workspace_bytes(M, N, K) exceeds that size is rejected with
 * MXFP4_ERR_WORKSPACE.  Nothing is allocated or freed.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress).  The address is kept for the process:
 *     resetting the device (cudaDeviceReset) while the library is in use is
 *     not supported.
 *   - All calls share the one array and it keeps the last call's contents
 *     (no call needs it cleared); calls that overlap on the GPU — on
 *     different streams, or from several host threads without ordering —
 *     race on it.
 */
MXFP4_API mxfp4_status mxfp4_gemm_noalloc(const void* a_bf16_dev, int lda, const void* w_packed_dev,
                                          const void* bias_dev, void* out_dev, int ldo, int M, int N, int K,
                                          void* stream);
MXFP4_API size_t mxfp4_gemm_noalloc_max_scratch_bytes(void);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * words on the current device.  Returns MXFP4_ERR_TIMEOUT if a kernel gave
 * up a bounded wait since the last call, MXFP4_OK otherwise (or
 * MXFP4_ERR_CUDA if the synchronisation itself failed).
 */
MXFP4_API mxfp4_status mxfp4_get_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_H */
