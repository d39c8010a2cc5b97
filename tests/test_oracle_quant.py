"""Pins of the oracle's per-1x32 quantizer (CPU only).

The oracle uses frexp for the shared exponent and a per-binade half-to-even
rint for the elements.  These tests pin it against an exact-rational brute
force (search for the exponent with 4 <= amax/2**E < 8, argmin over the eight
E2M1 magnitudes with ties to the even code) and against hand-derived cases:
every rounding tie, saturation, power-of-two boundaries, zero and subnormal
blocks, signed zeros and the nibble order.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import mxfp4_ref as ref
from mxfp4_quantized_gemm_gb300 import synth

GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2),
        Fraction(3), Fraction(4), Fraction(6)]


def brute_block(vals):
    """Exact-rational quantization of one block of float values."""
    fr = [Fraction(float(v)) for v in vals]
    amax = max(abs(v) for v in fr)
    if amax == 0:
        E = -127
    else:
        E = 200
        while amax < 4 * Fraction(2) ** E:
            E -= 1
        E = max(-127, min(127, E))
    codes = []
    for x, v in zip(vals, fr):
        q = abs(v) / Fraction(2) ** E
        best = None
        for idx, gv in enumerate(GRID):
            d = abs(q - gv)
            if best is None or d < best[0] or (d == best[0] and idx % 2 == 0):
                best = (d, idx)
        sign = 8 if np.signbit(x) else 0
        codes.append(best[1] | sign)
    return E + 127, codes


def oracle_block(vals):
    c, s = ref.quantize_mxfp4(np.asarray(vals, dtype=np.float64)[None, :])
    nib = ref.unpack_codes(c, len(vals))[0]
    return int(s[0, 0]), [int(v) for v in nib]


def test_random_blocks_match_brute_force():
    g = np.random.default_rng(5)
    bits = synth.activations(64, 32 * 12, seed=9, outlier_frac=0.05)
    x = ref.bf16_bits_to_f64(bits)
    # widen the exponent range so the clamps are reached too
    x = x * np.ldexp(1.0, g.integers(-140, 120, size=(64, 1)))
    x = ref.bf16_bits_to_f64(ref.f64_to_bf16_bits(x))
    codes, scales = ref.quantize_mxfp4(x)
    nib = ref.unpack_codes(codes, x.shape[1])
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 32):
            s, c = brute_block(x[r, 32 * b:32 * b + 32])
            assert int(scales[r, b]) == s, (r, b)
            assert [int(v) for v in nib[r, 32 * b:32 * b + 32]] == c, (r, b)


def test_edge_rows_match_brute_force():
    for K in (64, 320):
        for row in synth.edge_rows(K, seed=3):
            x = ref.bf16_bits_to_f64(row)
            codes, scales = ref.quantize_mxfp4(x[None, :])
            nib = ref.unpack_codes(codes, K)[0]
            for b in range(K // 32):
                s, c = brute_block(x[32 * b:32 * b + 32])
                assert int(scales[0, b]) == s
                assert [int(v) for v in nib[32 * b:32 * b + 32]] == c


def test_scaled_amax_lands_in_4_to_8():
    g = np.random.default_rng(6)
    x = g.standard_normal((200, 256)) * np.ldexp(1.0, g.integers(-100, 100, size=(200, 1)))
    _, scales = ref.quantize_mxfp4(x)
    amax = np.abs(x.reshape(200, 8, 32)).max(axis=2)
    r = amax / np.ldexp(1.0, scales.astype(np.int64) - 127)
    assert np.all((r >= 4) & (r < 8))


@pytest.mark.parametrize("E", [-120, -3, 0, 5, 120])
@pytest.mark.parametrize("top", [4.0, 6.0])
def test_round_trip_of_representable_blocks(E, top):
    g = np.random.default_rng(E + 1000)
    codes = g.integers(0, 16, size=32)
    vals = ref.e2m1_decode(codes)
    vals = np.clip(vals, -top, top)
    vals[3] = top
    x = np.ldexp(vals, E)
    s, c = oracle_block(x)
    assert s == E + 127
    assert np.array_equal(ref.e2m1_decode(c) * 2.0 ** E, x)


TIES = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}


@pytest.mark.parametrize("E", [-10, 0, 3])
def test_every_tie_goes_to_even_code(E):
    for t, code in TIES.items():
        block = np.zeros(32)
        block[0] = 4.0
        block[1] = t
        block[2] = -t
        s, c = oracle_block(np.ldexp(block, E))
        assert s == E + 127
        assert c[1] == code and c[2] == code | 8, t


def test_just_off_ties_round_to_nearest():
    for t, code in TIES.items():
        block = np.zeros(32)
        block[0] = 4.0
        block[1] = t * (1 + 2 ** -7)
        block[2] = t * (1 - 2 ** -7)
        _, c = oracle_block(block)
        grid = [float(v) for v in GRID]
        up = min(range(8), key=lambda i: abs(grid[i] - block[1]))
        dn = min(range(8), key=lambda i: abs(grid[i] - block[2]))
        assert c[1] == up and c[2] == dn


def test_saturation_beyond_six():
    block = np.array([7.0, 6.5, 7.5, 7.96875, -6.25, -7.96875] + [0.0] * 26)
    s, c = oracle_block(block)
    assert s == 127 + 0       # floor(log2 7.97) - 2 = 0
    assert c[:6] == [7, 7, 7, 7, 15, 15]


@pytest.mark.parametrize("k", [-126, -20, 0, 5, 100, 127])
def test_power_of_two_boundaries(k):
    block = np.zeros(32)
    block[7] = np.ldexp(1.0, k)
    s, c = oracle_block(block)
    assert s == max(k + 125, 0)
    if k + 125 >= 0:
        assert c[7] == 6                  # 2**k / 2**(k-2) = 4
    else:                                 # clamped scale 2**-127: 2**(k+127)
        assert c[7] == {1.0: 2, 2.0: 4}[2.0 ** (k + 127)]
    below = ref.bf16_bits_to_f64(np.uint16(((k + 127) << 7) - 1))
    block[7] = below
    s, c = oracle_block(block)
    assert s == max(k + 124, 0)
    if k + 124 >= 0:
        assert c[7] == 7                  # 8 * (1 - 2**-8) saturates to 6


def test_zero_and_subnormal_blocks_get_smallest_scale():
    s, c = oracle_block(np.zeros(32))
    assert s == 0 and c == [0] * 32
    s, c = oracle_block(-np.zeros(32))
    assert s == 0 and c == [8] * 32
    sub = ref.bf16_bits_to_f64(np.arange(1, 33, dtype=np.uint16))
    s, c = oracle_block(sub)
    assert s == 0
    # 2**-127 scale: the largest subnormal 32 * 2**-133 = 2**-128 is 0.5
    assert c[31] == 1


def test_negative_values_rounding_to_zero_keep_sign():
    block = np.zeros(32)
    block[0] = 4.0
    block[1] = -0.2
    block[2] = 0.2
    _, c = oracle_block(block)
    assert c[1] == 8 and c[2] == 0


def test_nibble_order_low_first():
    x = np.zeros((1, 32))
    x[0, 0] = 4.0      # code 6
    x[0, 1] = -1.0     # code 10
    codes, _ = ref.quantize_mxfp4(x)
    assert codes[0, 0] == 6 | (10 << 4)


def test_partial_last_block_is_zero_padded():
    g = np.random.default_rng(8)
    x = g.standard_normal((3, 40))
    c40, s40 = ref.quantize_mxfp4(x)
    xp = np.zeros((3, 64))
    xp[:, :40] = x
    c64, s64 = ref.quantize_mxfp4(xp)
    assert np.array_equal(s40, s64)
    assert np.array_equal(c40, c64[:, :20])


def test_nonfinite_block_reading():
    block = np.zeros(32)
    block[0] = np.inf
    block[1] = 3.0
    s, c = oracle_block(block)
    assert s == 0xFF and c == [0] * 32
