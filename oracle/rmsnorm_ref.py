"""Plain CPU oracle for the fused RMSNorm -> MXFP4 activation producer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA path.

The pages let the GEMM take its activations already quantized and name a
fused RMSNorm as one producer of that (codes, scales) tuple (sglang PR #39598
blog analysis, section 2, apply_weights), but print neither the
normalization nor its rounding.  The plainest reading, used here:

* RMSNorm as defined by Zhang and Sennrich (2019), with the usual epsilon
  inside the root:  y_i = h_i / sqrt(mean_j(h_j**2) + eps) * gamma_i;
* the optional fused residual add first forms h = bf16(x + residual) and
  that sum is also the updated residual;
* y is rounded once to bfloat16, and those bfloat16 values are quantized per
  1x32 exactly as a separate quantizer would quantize them
  (``mxfp4_ref.quantize_mxfp4``), so the fused producer equals the unfused
  "RMSNorm to bf16, then per_1x32_f4_quant" pipeline.

Everything is float64; eps is taken as the float32 value the kernel receives.
"""

from __future__ import annotations

import numpy as np

from . import mxfp4_ref as ref


def add_residual(x_bits, res_bits) -> np.ndarray:
    """h = bf16(x + residual): the exact sum of two bf16 values, rounded once."""
    return ref.f64_to_bf16_bits(ref.bf16_bits_to_f64(x_bits) + ref.bf16_bits_to_f64(res_bits))


def rmsnorm_f64(h_bits, gamma_bits, eps: float) -> np.ndarray:
    """Exact-as-float64 RMSNorm of the rows of h [rows, K] (bf16 bits)."""
    h = ref.bf16_bits_to_f64(h_bits)
    g = ref.bf16_bits_to_f64(gamma_bits)
    e = float(np.float32(eps))
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        ms = np.mean(h * h, axis=1, keepdims=True)
        return h / np.sqrt(ms + e) * g[None, :]


def rmsnorm_quant(x_bits, gamma_bits, eps: float, res_bits=None) -> dict:
    """The fused producer's results for x [rows, K] (bf16 bits):

    ``h``      bf16 bits of the normalized input (x, or x + residual rounded),
               which is also the updated residual;
    ``y_exact`` float64 RMSNorm of h;
    ``y``      its bf16 bits (one rounding);
    ``codes``, ``scales``  per-1x32 MXFP4 quantization of y (row-major).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    h = x_bits if res_bits is None else add_residual(x_bits, res_bits)
    y_exact = rmsnorm_f64(h, gamma_bits, eps)
    y = ref.f64_to_bf16_bits(y_exact)
    codes, scales = ref.quantize_mxfp4(ref.bf16_bits_to_f64(y))
    return {"h": h, "y_exact": y_exact, "y": y, "codes": codes, "scales": scales}
