"""Shared test plumbing: device buffers, calls through the C ABI, and the
oracle comparison with the bf16 tolerance.

Tolerance (floating point outputs): |out - ref| <= 2 ulp(ref), ref being the
float64 oracle rounded once to bf16 and ulp(r) = 2**(floor(log2|r|) - 7) for
normal r, 2**-133 below the normal range.  An output that misses it passes
only under the fp32-summation allowance n_acc * 2**-24 * sum_k |a_k w_k|
(recursive-summation error bound; n_acc = fp32 additions on the output's
reduction path), and such outputs are counted: by default at most
2 + n/10000 of n outputs may use it.  NaN/Inf never pass unless the reference is
NaN/Inf too.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import mxfp4_ref as ref
from oracle import tile_layout as tl
from mxfp4_quantized_gemm_gb300 import synth


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return synth.bf16_tensor(bits).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def empty_u8(n: int) -> torch.Tensor:
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device="cuda")


def gemm_workspace(capi, n: int) -> torch.Tensor:
    """A GEMM workspace as a caller would set one up: arbitrary contents
    (filled with 0xA5 here; the GEMM needs no initialization)."""
    return torch.full((max(int(n), 1),), 0xA5, dtype=torch.uint8, device="cuda")


def pack_weights(capi, codes: np.ndarray, scales: np.ndarray, K: int) -> torch.Tensor:
    """codes [B?, N, K/2], scales [B?, N, ceil(K/32)] -> packed device buffer."""
    if codes.ndim == 2:
        codes, scales = codes[None], scales[None]
    B, N = codes.shape[0], codes.shape[1]
    packed = empty_u8(capi.mxfp4_packed_weight_bytes(B, N, K))
    capi.mxfp4_pack_weights(dev_u8(codes), dev_u8(scales), B, N, K, packed)
    return packed


def ulp_bf16(r: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(r, dtype=np.float64))
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    u = np.ldexp(1.0, e - 1 - 7)
    return np.where(a >= 2.0 ** -126, u, 2.0 ** -133)


def allowance_budget(n: int, K: int | None = None) -> int:
    """Outputs that may need the summation allowance: near-cancelling sums are
    rare.  Short sums need it too (an output whose exact value cancels to a
    small fraction of its terms' magnitudes misses 2 ulp after a single fp32
    rounding of a partial sum), so K does not change the budget; the count is
    reported at the end of the session."""
    return 2 + n // 10000


# Every comparison's statistics, in order, for the end-of-session report
# (conftest.py prints how many outputs passed only under the allowance).
ALLOWANCE_LOG: list[dict] = []


def check_close(out_bits: np.ndarray, acc: np.ndarray, absdot: np.ndarray, n_acc: int,
                max_allowance: int | None = -1, what: str = "", K: int | None = None) -> dict:
    """Compare bf16 outputs against the float64 oracle; return statistics
    (also appended to ALLOWANCE_LOG).  K, when given, sets the allowance
    budget (none for K <= 512)."""
    out = ref.bf16_bits_to_f64(out_bits)
    refb = ref.bf16_bits_to_f64(ref.f64_to_bf16_bits(acc))
    ref_nonfinite = ~np.isfinite(refb)
    bad_nonfinite = (~np.isfinite(out)) & ~ref_nonfinite
    assert not bad_nonfinite.any(), f"{what}: {int(bad_nonfinite.sum())} unexpected NaN/Inf outputs"
    nan_ref = np.isnan(refb)
    assert np.isnan(out[nan_ref]).all(), f"{what}: {int((~np.isnan(out[nan_ref])).sum())} outputs are not NaN " \
        "where the oracle's are (a 0xFF scale in a contributing block)"
    inf_ref = np.isinf(refb)
    assert np.array_equal(out[inf_ref], refb[inf_ref]), f"{what}: an overflowing output is not the oracle's Inf"
    fin = ~ref_nonfinite
    err = np.abs(out - refb)
    tol = 2.0 * ulp_bf16(refb)
    strict = (err <= tol) | ~fin
    allow = tol + n_acc * 2.0 ** -24 * absdot
    loose = (err <= allow) | ~fin
    n_fail = int((~loose).sum())
    n_allow = int((loose & ~strict).sum())
    if n_fail:
        idx = np.argwhere(~loose)[:5]
        details = [(tuple(int(v) for v in i), float(out[tuple(i)]), float(refb[tuple(i)]), float(acc[tuple(i)]))
                   for i in idx]
        raise AssertionError(f"{what}: {n_fail} outputs beyond tolerance, e.g. (index, out, ref, exact) {details}")
    ratio = np.where(fin, err / np.maximum(ulp_bf16(refb), 1e-300), 0.0)
    stats = {"what": what, "K": K, "max_ulp": float(ratio.max(initial=0.0)), "n_allowance": n_allow,
             "n": int(out.size)}
    ALLOWANCE_LOG.append(stats)
    if max_allowance == -1:
        max_allowance = allowance_budget(int(out.size), K)
    if max_allowance is not None:
        assert n_allow <= max_allowance, f"{what}: {n_allow} outputs needed the fp32 summation allowance"
    return stats


def sample_rows(M: int, seed: int = 0, n_random: int = 48, boundary_stride: int = 4) -> np.ndarray:
    """First, last, rows around every `boundary_stride`-th 128-row tile boundary, seeded random rows."""
    rows = {0, M - 1}
    for t in range(128, M, 128 * boundary_stride):
        rows.update({t - 1, t, t + 1})
    g = np.random.default_rng(seed)
    rows.update(int(v) for v in g.integers(0, M, size=min(n_random, M)))
    return np.array(sorted(r for r in rows if 0 <= r < M))


def oracle_gemm_rows(x_bits: np.ndarray, rows: np.ndarray, w_codes, w_scales, K: int, bias_bits=None,
                     n_chunk: int = 8192):
    """Oracle (quantize, then dequantized matmul) on the selected activation rows."""
    x = ref.bf16_bits_to_f64(x_bits[rows])
    a_c, a_s = ref.quantize_mxfp4(x)
    N = w_codes.shape[0]
    acc = np.empty((len(rows), N))
    mag = np.empty((len(rows), N))
    bias = ref.bf16_bits_to_f64(bias_bits) if bias_bits is not None else None
    for n0 in range(0, N, n_chunk):
        n1 = min(N, n0 + n_chunk)
        a, m = ref.mxfp4_gemm_f64(a_c, a_s, w_codes[n0:n1], w_scales[n0:n1], K,
                                  None if bias is None else bias[n0:n1])
        acc[:, n0:n1] = a
        mag[:, n0:n1] = m
    return acc, mag


def tiled_from_oracle(codes: np.ndarray, scales: np.ndarray, K: int):
    """Split the oracle's packed image into (codes region, scales region)."""
    packed = tl.pack(codes, scales, K)
    cb = tl.code_bytes(codes.shape[0], K)
    return packed[:cb], packed[cb:]
