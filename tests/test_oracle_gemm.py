"""Pins of the oracle's W4A4 GEMM and A16WFP4 batched matmul (CPU only).

Checked against exact integer/rational brute force on tiny shapes (2*E2M1
values are integers and E8M0 scales are powers of two, so every product is an
exact rational), against an integer matmul where the operands reduce to
integers, and against special cases with a known answer.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import mxfp4_ref as ref
from mxfp4_quantized_gemm_gb300 import synth
from test_oracle_formats import bf16_bits_exact, e2m1_from_bits


def exact_gemm(a_codes, a_scales, w_codes, w_scales, K, bias_bits=None):
    M, N = a_codes.shape[0], w_codes.shape[0]
    an = ref.unpack_codes(a_codes, K)
    wn = ref.unpack_codes(w_codes, K)
    out = np.zeros((M, N), dtype=np.uint16)
    exact = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                sa = int(a_scales[m, k // 32]) - 127
                sw = int(w_scales[n, k // 32]) - 127
                acc += e2m1_from_bits(int(an[m, k])) * e2m1_from_bits(int(wn[n, k])) * Fraction(2) ** (sa + sw)
            if bias_bits is not None:
                acc += Fraction(float(ref.bf16_bits_to_f64(bias_bits[n])))
            exact[m][n] = acc
            out[m, n] = bf16_bits_exact(acc)
    return out, exact


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 64), (6, 4, 96), (5, 6, 128)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_matches_exact_brute_force(M, N, K, with_bias):
    seed = M * 100 + N * 10 + K
    a_c = synth.weight_codes(M, K, seed, 11)
    a_s = synth.weight_scales(M, K, -8, 2, seed, 12)
    w_c = synth.weight_codes(N, K, seed, 13)
    w_s = synth.weight_scales(N, K, -6, 0, seed, 14)
    b = synth.bias(N, seed, 15) if with_bias else None
    want, exact = exact_gemm(a_c, a_s, w_c, w_s, K, b)
    bias64 = ref.bf16_bits_to_f64(b) if with_bias else None
    got = ref.mxfp4_gemm(a_c, a_s, w_c, w_s, K, bias64)
    acc, _ = ref.mxfp4_gemm_f64(a_c, a_s, w_c, w_s, K, bias64)
    # non-zero results: bits agree; exact zeros may carry either sign in float64
    nz = np.array([[e != 0 for e in row] for row in exact])
    assert np.array_equal(got[nz], want[nz])
    assert np.all((got[~nz] & 0x7FFF) == 0)
    for m in range(M):
        for n in range(N):
            assert Fraction(float(acc[m, n])) == exact[m][n]


def test_quant_then_gemm_matches_brute_force():
    K = 96
    x = ref.bf16_bits_to_f64(synth.activations(4, K, seed=4, outlier_frac=0.05))
    w_c = synth.weight_codes(3, K, 4, 13)
    w_s = synth.weight_scales(3, K, -8, 2, 4, 14)
    a_c, a_s = ref.quantize_mxfp4(x)
    want, _ = exact_gemm(a_c, a_s, w_c, w_s, K)
    acc, _ = ref.quant_then_gemm(x, w_c, w_s, K)
    got = ref.f64_to_bf16_bits(acc)
    assert np.array_equal(got & 0x7FFF, want & 0x7FFF)


def test_zero_activation_gives_bias_exactly():
    K, N = 256, 40
    a_c, a_s = ref.quantize_mxfp4(np.zeros((3, K)))
    w_c = synth.weight_codes(N, K, 1)
    w_s = synth.weight_scales(N, K, -6, 0, 1)
    b = synth.bias(N, 1)
    got = ref.mxfp4_gemm(a_c, a_s, w_c, w_s, K, ref.bf16_bits_to_f64(b))
    assert np.array_equal(got, np.broadcast_to(b, got.shape))


def test_single_nonzero_product():
    K = 128
    a_c = np.zeros((2, K // 2), np.uint8)
    w_c = np.zeros((3, K // 2), np.uint8)
    a_s = np.full((2, K // 32), 120, np.uint8)
    w_s = np.full((3, K // 32), 130, np.uint8)
    a_c[1, 40] = 0x70          # element 81 of row 1 = code 7 (6.0)
    w_c[2, 40] = 0xB0          # element 81 of row 2 = code 11 (-1.5)
    got = ref.bf16_bits_to_f64(ref.mxfp4_gemm(a_c, a_s, w_c, w_s, K))
    want = np.zeros((2, 3))
    want[1, 2] = 6.0 * -1.5 * 2.0 ** (120 - 127 + 130 - 127)
    assert np.array_equal(got, want)


def test_integer_operands_reduce_to_integer_matmul():
    g = np.random.default_rng(3)
    M, N, K = 9, 11, 256
    ai = g.integers(-1, 2, size=(M, K))
    wi = g.integers(-1, 2, size=(N, K))
    enc = {0: 0, 1: 2, -1: 10}             # E2M1 codes of 0, 1.0, -1.0
    def pack(v):
        c = np.vectorize(enc.get)(v).astype(np.uint8)
        return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    ones_a = np.full((M, K // 32), 127, np.uint8)
    ones_w = np.full((N, K // 32), 127, np.uint8)
    got = ref.bf16_bits_to_f64(ref.mxfp4_gemm(pack(ai), ones_a, pack(wi), ones_w, K))
    assert np.array_equal(got, (ai @ wi.T).astype(np.float64))


def test_nan_scale_poisons_only_its_row():
    K = 64
    a_c = synth.weight_codes(2, K, 5, 1)
    a_s = np.full((2, 2), 127, np.uint8)
    a_s[1, 1] = 0xFF
    w_c = synth.weight_codes(3, K, 5, 2)
    w_s = np.full((3, 2), 127, np.uint8)
    out = ref.bf16_bits_to_f64(ref.mxfp4_gemm(a_c, a_s, w_c, w_s, K))
    assert np.all(np.isfinite(out[0])) and np.all(np.isnan(out[1]))


def test_bmm_matches_exact_brute_force_and_layouts():
    B, M, N, K = 3, 4, 5, 64
    xb = synth.bmm_activations(B, M, K, seed=2)
    w_c = synth.weight_codes(N, K, 2, 7, batch=B)
    w_s = synth.weight_scales(N, K, -6, 0, 2, 8, batch=B)
    x = ref.bf16_bits_to_f64(xb)
    got = ref.a16wfp4_bmm(x, w_c, w_s, K)
    got_mbn = ref.a16wfp4_bmm(x, w_c, w_s, K, batch_major=True)
    assert got.shape == (B, M, N) and got_mbn.shape == (M, B, N)
    for b in range(B):
        wn = ref.unpack_codes(w_c[b], K)
        for m in range(M):
            for n in range(N):
                acc = Fraction(0)
                for k in range(K):
                    acc += (Fraction(float(x[b, m, k])) * e2m1_from_bits(int(wn[n, k]))
                            * Fraction(2) ** (int(w_s[b, n, k // 32]) - 127))
                if acc != 0:
                    assert got[b, m, n] == bf16_bits_exact(acc)
                assert got_mbn[m, b, n] == got[b, m, n]


def _permute_blocks(codes, scales, perm):
    """Reorder the 32-element K blocks of [R, K/2] codes and [R, K/32] scales."""
    R, nb = scales.shape
    c = codes.reshape(R, nb, 16)[:, perm, :].reshape(R, nb * 16)
    return np.ascontiguousarray(c), np.ascontiguousarray(scales[:, perm])


def test_consistent_permutations_commute_with_the_gemm():
    """At a size past brute force: reordering the K blocks of both operands
    the same way leaves every sum unchanged (each product is an exact dyadic
    rational and the sums stay exact in float64 here), and reordering the
    weight rows reorders the output columns.  A transposed operand, a wrong
    block index or a scale read from the wrong row breaks one of them."""
    M, N, K = 7, 40, 2048
    g = np.random.default_rng(12)
    a_c = synth.weight_codes(M, K, 12, 1)
    a_s = synth.weight_scales(M, K, -4, 2, 12, 2)
    w_c = synth.weight_codes(N, K, 12, 3)
    w_s = synth.weight_scales(N, K, -8, 0, 12, 4)
    base = ref.mxfp4_gemm_f64(a_c, a_s, w_c, w_s, K)[0]
    perm = g.permutation(K // 32)
    pa = _permute_blocks(a_c, a_s, perm)
    pw = _permute_blocks(w_c, w_s, perm)
    assert np.array_equal(ref.mxfp4_gemm_f64(*pa, *pw, K)[0], base)
    rows = g.permutation(N)
    assert np.array_equal(ref.mxfp4_gemm_f64(a_c, a_s, w_c[rows], w_s[rows], K)[0], base[:, rows])
    # permuting only one operand's blocks changes the result (the test can fail)
    assert not np.array_equal(ref.mxfp4_gemm_f64(*pa, w_c, w_s, K)[0], base)
