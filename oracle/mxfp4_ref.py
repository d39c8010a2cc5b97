"""Plain, slow CPU oracle for the MXFP4 block-scaled dense linear.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code, table or constant with the CUDA
path under ``mxfp4_quantized_gemm_gb300/csrc``.

Everything here is written in float64 numpy, straight from the definitions:

* E2M1 element codes (4 bits: sign, 2 exponent bits with bias 1, 1 mantissa
  bit) and E8M0 block scales (an unsigned biased exponent, 2**(e-127), with
  0xFF reserved for NaN), as in the OCP Microscaling (MX) v1.0 format
  definition.  The pages fix two of these facts themselves: the E8M0 byte
  0x7F is 1.0 and 0xFF is NaN (sglang PR #39598 blog analysis, section 2,
  ``_E8M0_ONE`` and the comment on padding activation scales).
* Per-1x32 quantization: one E8M0 scale per 32 consecutive K-elements of a
  row, codes packed two per byte into ``[rows, cols // 2]`` and scales shaped
  ``[rows, ceil(cols / 32)]`` (sglang PR #39598 blog analysis, section 2,
  ``_aiter_per_1x32_f4_quant_fake``).  The scale exponent is the OCP MX rule
  floor(log2(amax)) - 2 (2 being the largest exponent of E2M1), the element
  conversion is round-to-nearest-even with saturation at +-6.
* The W4A4 GEMM is "dequantize both operands, then matmul", the semantics the
  first page validates the kernel against ("[AMD] Add opt-in AITER ASM FP4
  GEMM for Quark dense linear", Accuracy Tests: identical to a separately
  dequantized FP4 reference), with the bias added after the product
  (blog analysis, section 2, ``apply_weights``) and one final rounding to
  bfloat16.
* The A16WFP4 batched matmul of "[AMD] [GLM5] use tuned MXFP4 kernels for MLA
  absorbed BMM" (Modifications): bf16 activations against FP4 weights with
  E8M0 scales, the V-up output written batch-major ``[M, B, N]``.

Readings where the pages are silent:

* nibble order: element 2j in the low nibble, element 2j+1 in the high nibble
  of byte j;
* an all-zero (or all-subnormal) block gets the smallest scale, byte 0x00
  (the clamp of the OCP exponent to the E8M0 range);
* the code of a zero or of a negative value that rounds to zero keeps the
  input's sign bit (so -0.0 encodes as 0x8);
* a block holding Inf or NaN gets scale 0xFF and codes 0;
* when K is not a multiple of 32, the missing elements of the last block are
  zeros;
* the split + cat epilogue, which the pages only name (blog analysis,
  section 2: a 5-tuple input requests the Triton-only fused "split + cat"
  epilogue, ``fused_gemm_afp4wfp4_split_cat``): the GEMM's bf16 result is
  viewed as H groups of s1 + s2 columns; each group's first s1 columns,
  followed by a caller tensor's s3 values for that row and group, form one
  output, its last s2 columns the other (``split_cat``).
"""

from __future__ import annotations

import numpy as np

BLOCK = 32                      # K-elements per E8M0 scale
E2M1_EMAX = 2                   # largest unbiased exponent of E2M1 (6 = 1.5 * 2**2)
E8M0_BIAS = 127
E8M0_NAN = 0xFF
# Magnitudes of the eight non-negative E2M1 codes 0..7 (code 8..15 = negatives).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


# --------------------------------------------------------------------------
# element formats
# --------------------------------------------------------------------------
def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (bit 3 = sign, bits 0..2 = magnitude index)."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    mag = E2M1_GRID[c & 7]
    return np.where(c & 8, -mag, mag)


def e8m0_decode(scale_bytes) -> np.ndarray:
    """2**(e - 127) for e in 0..254, NaN for 0xFF."""
    e = np.asarray(scale_bytes, dtype=np.int64)
    val = np.ldexp(1.0, e - E8M0_BIAS)
    return np.where(e == E8M0_NAN, np.nan, val)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values once, to nearest-even, onto the bfloat16 grid.

    bfloat16 has an 8-bit significand and float32's exponent range: normal
    numbers >= 2**-126 are rounded to a quantum of 2**(floor(log2|x|) - 7),
    smaller ones to the subnormal quantum 2**-133.  Results beyond the largest
    finite bfloat16 become +-Inf; NaN stays NaN; the sign of zero is kept.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    nan = np.isnan(x)
    a_fin = np.where(np.isfinite(a), a, 0.0)
    _, e = np.frexp(a_fin)                      # a = m * 2**e, m in [0.5, 1)
    q_exp = np.maximum(e - 8, -133)              # quantum exponent
    n = np.rint(np.ldexp(a_fin, -q_exp))         # half-to-even on the quantum count
    mag = np.ldexp(n, q_exp)
    mag = np.where(np.isinf(a) | (mag > BF16_MAX), np.inf, mag)
    bits = (mag.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.signbit(x), bits | np.uint16(0x8000), bits)
    bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


# --------------------------------------------------------------------------
# per-1x32 quantization (OCP MX conversion rule)
# --------------------------------------------------------------------------
def _round_e2m1_magnitude(v: np.ndarray) -> np.ndarray:
    """Index 0..7 of the E2M1 magnitude nearest to |v|, ties to the even code.

    Saturating conversion: |v| above 6 maps to 6.  Within each binade the
    E2M1 grid is uniform (quantum 0.5 below 2, 1 in [2, 4), 2 in [4, 6]), so
    nearest-even rounding is a half-to-even rint of |v| / quantum.
    """
    a = np.minimum(np.abs(v), 6.0)
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    q = np.rint(a / quantum) * quantum
    return np.searchsorted(E2M1_GRID, q)


def quantize_mxfp4(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-1x32 MXFP4 quantization of a float matrix ``x[rows, K]`` (K even).

    Returns ``(codes uint8 [rows, K//2], scales uint8 [rows, ceil(K/32)])``.
    For every block of 32 elements along K:
      1. amax = max |x_i| over the block;
      2. shared exponent E = floor(log2 amax) - 2, clamped to the E8M0 range
         [-127, 127] (amax = 0 clamps to -127); the scale byte is E + 127;
      3. each element is divided by 2**E and rounded to the nearest E2M1 value
         (ties to even, saturating at 6); the code keeps the input's sign bit.
    """
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2 or x.shape[1] % 2:
        raise ValueError("x must be [rows, K] with K even")
    rows, K = x.shape
    nb = -(-K // BLOCK)
    xp = np.zeros((rows, nb * BLOCK), dtype=np.float64)
    xp[:, :K] = x
    blk = xp.reshape(rows, nb, BLOCK)

    finite = np.isfinite(blk).all(axis=2)
    amax = np.abs(np.where(np.isfinite(blk), blk, 0.0)).max(axis=2)
    _, ex = np.frexp(amax)                       # amax = m * 2**ex, m in [0.5, 1)
    floor_log2 = ex - 1
    E = np.where(amax > 0, floor_log2 - E2M1_EMAX, -E8M0_BIAS)
    E = np.clip(E, -E8M0_BIAS, E8M0_BIAS)
    scales = np.where(finite, E + E8M0_BIAS, E8M0_NAN).astype(np.uint8)

    v = np.ldexp(np.where(finite[:, :, None], blk, 0.0), -E[:, :, None])
    mag = _round_e2m1_magnitude(v)
    sign = np.signbit(blk) & finite[:, :, None]
    codes4 = (mag | (sign.astype(np.int64) << 3)).reshape(rows, nb * BLOCK)[:, :K]
    codes = (codes4[:, 0::2] | (codes4[:, 1::2] << 4)).astype(np.uint8)
    return codes, scales


def unpack_codes(codes, K: int) -> np.ndarray:
    """[rows, K//2] packed bytes -> [rows, K] 4-bit codes (low nibble first)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty((c.shape[0], K), dtype=np.uint8)
    out[:, 0::2] = c[:, : K // 2] & 0xF
    out[:, 1::2] = c[:, : K // 2] >> 4
    return out


def dequantize_mxfp4(codes, scales, K: int) -> np.ndarray:
    """deq(c, s) = e2m1(c) * 2**(s - 127) for every element, float64 [rows, K]."""
    vals = e2m1_decode(unpack_codes(codes, K))
    s = e8m0_decode(np.asarray(scales)).repeat(BLOCK, axis=1)[:, :K]
    return vals * s


# --------------------------------------------------------------------------
# W4A4 GEMM and A16WFP4 batched matmul
# --------------------------------------------------------------------------
def mxfp4_gemm_f64(a_codes, a_scales, w_codes, w_scales, K: int, bias=None):
    """Unrounded result sum_k deq(A)[m,k] * deq(W)[n,k] (+ bias[n]), float64.

    Also returns sum_k |deq(A)[m,k] * deq(W)[n,k]|, the magnitude that bounds
    the rounding error of any fp32 summation order (used by the tests).
    ``bias`` is a float64 vector of bfloat16 values or None.
    """
    a = dequantize_mxfp4(a_codes, a_scales, K)
    w = dequantize_mxfp4(w_codes, w_scales, K)
    acc = a @ w.T
    absdot = np.abs(a) @ np.abs(w).T
    if bias is not None:
        acc = acc + np.asarray(bias, dtype=np.float64)[None, :]
    return acc, absdot


def mxfp4_gemm(a_codes, a_scales, w_codes, w_scales, K: int, bias=None) -> np.ndarray:
    """out = bf16_RNE(sum_k deq(A)[m,k] * deq(W)[n,k] + bias[n]) as bf16 bits."""
    acc, _ = mxfp4_gemm_f64(a_codes, a_scales, w_codes, w_scales, K, bias)
    return f64_to_bf16_bits(acc)


def quant_then_gemm(x, w_codes, w_scales, K: int, bias=None):
    """The dense linear as a whole: quantize bf16 rows, then the W4A4 GEMM."""
    a_codes, a_scales = quantize_mxfp4(x)
    return mxfp4_gemm_f64(a_codes, a_scales, w_codes, w_scales, K, bias)


def a16wfp4_bmm_f64(x, w_codes, w_scales, K: int):
    """out[b, m, n] = sum_k x[b, m, k] * deq(W)[b, n, k], float64, plus |.|-sum.

    ``x`` is float64 [B, M, K] holding bfloat16 values.
    """
    x = np.asarray(x, dtype=np.float64)
    B = x.shape[0]
    outs, mags = [], []
    for b in range(B):
        w = dequantize_mxfp4(w_codes[b], w_scales[b], K)
        outs.append(x[b] @ w.T)
        mags.append(np.abs(x[b]) @ np.abs(w).T)
    return np.stack(outs), np.stack(mags)


def a16wfp4_bmm(x, w_codes, w_scales, K: int, batch_major: bool = False) -> np.ndarray:
    """bf16 bits of the batched product; ``batch_major`` gives [M, B, N] (V-up)."""
    acc, _ = a16wfp4_bmm_f64(x, w_codes, w_scales, K)
    bits = f64_to_bf16_bits(acc)
    return np.ascontiguousarray(bits.transpose(1, 0, 2)) if batch_major else bits


def split_cat(y_bits, z_bits, s1: int, s2: int):
    """The split + cat epilogue on the GEMM's bf16 result (a reading: the pages
    give only the name, blog analysis section 2).

    ``y_bits`` [M, H * (s1 + s2)] bf16 bits, ``z_bits`` [M, H, s3] bf16 bits.
    Returns (cat [M, H, s1 + s3], split [M, H, s2]): for every row m and group
    h, cat[m, h] = y[m, h-th group's first s1 columns] followed by z[m, h],
    split[m, h] = the group's last s2 columns.  Pure data movement.
    """
    y = np.asarray(y_bits, dtype=np.uint16)
    z = np.asarray(z_bits, dtype=np.uint16)
    M, N = y.shape
    G = s1 + s2
    H = N // G
    assert H * G == N and z.shape[:2] == (M, H)
    s3 = z.shape[2]
    cat = np.empty((M, H, s1 + s3), dtype=np.uint16)
    split = np.empty((M, H, s2), dtype=np.uint16)
    for h in range(H):
        group = y[:, h * G:(h + 1) * G]
        cat[:, h, :s1] = group[:, :s1]
        cat[:, h, s1:] = z[:, h, :]
        split[:, h, :] = group[:, s1:]
    return cat, split
