"""Pins of the oracle's element formats and bf16 rounding (CPU only).

Each check compares the oracle with something other than itself: the bit-field
definition of E2M1/E8M0, exact rationals, torch's own float32->bfloat16
conversion, or facts the pages state (tests/golden/page_facts.json).
"""

import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mxfp4_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def e2m1_from_bits(code: int) -> Fraction:
    """E2M1 from its fields: sign s, exponent e (bias 1), mantissa m."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -mag if s else mag


def test_e2m1_table_matches_bit_fields():
    got = ref.e2m1_decode(np.arange(16))
    for c in range(16):
        assert Fraction(float(got[c])) == e2m1_from_bits(c), c
    # code 8 is negative zero
    assert math.copysign(1.0, float(got[8])) == -1.0


def test_e8m0_table():
    got = ref.e8m0_decode(np.arange(256))
    for e in range(255):
        assert Fraction(float(got[e])) == Fraction(2) ** (e - 127), e
    assert math.isnan(got[255])


def test_page_facts_e8m0():
    facts = json.load(open(GOLDEN))
    assert ref.e8m0_decode(facts["e8m0_one"]["byte"]) == facts["e8m0_one"]["value"]
    assert math.isnan(ref.e8m0_decode(facts["e8m0_nan"]["byte"]))


def test_page_facts_quant_shapes():
    facts = json.load(open(GOLDEN))
    for rows, cols, cshape, sshape in facts["quant_output_shapes"]["cases"]:
        x = np.zeros((rows, cols))
        codes, scales = ref.quantize_mxfp4(x)
        assert list(codes.shape) == cshape and codes.dtype == np.uint8
        assert list(scales.shape) == sshape and scales.dtype == np.uint8


def test_page_facts_gemm_shape():
    f = json.load(open(GOLDEN))["gemm_output_shape"]
    M, N, K = f["M"], f["N"], f["K"]
    a_c, a_s = ref.quantize_mxfp4(np.zeros((M, K)))
    w_c = np.zeros((N, K // 2), np.uint8)
    w_s = np.full((N, K // 32), 127, np.uint8)
    assert list(ref.mxfp4_gemm(a_c, a_s, w_c, w_s, K).shape) == f["out"]


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------
BF16_MAX = Fraction(2 ** 8 - 1, 2 ** 7) * Fraction(2) ** 127


def bf16_bits_exact(q: Fraction, negative_zero=False) -> int:
    """Round a rational to bfloat16, nearest-even, using only integer arithmetic."""
    if q == 0:
        return 0x8000 if negative_zero else 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    qe = max(e - 7, -133)
    n = a / Fraction(2) ** qe
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * Fraction(2) ** qe
    if val > BF16_MAX:
        return sign | 0x7F80
    bits = struct.unpack("<I", struct.pack("<f", float(val)))[0] >> 16
    return sign | bits


def test_bf16_rounding_matches_torch_on_float32_values():
    g = np.random.default_rng(11)
    raw = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x32 = raw.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    # add exact ties: a bf16 value plus half a quantum
    base = (g.integers(0, 2 ** 16, size=5000).astype(np.uint32) << 16) | 0x8000
    x32 = np.concatenate([x32, base.view(np.float32)])
    x32 = x32[np.isfinite(x32)]
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = ref.f64_to_bf16_bits(x32.astype(np.float64))
    # torch may keep NaN payloads differently; there are none here
    assert np.array_equal(got, want)


def test_bf16_rounding_matches_exact_rationals():
    g = np.random.default_rng(12)
    xs = list(g.standard_normal(3000) * 10.0 ** g.integers(-40, 38, 3000))
    xs += [2.0 ** -133 * 0.5, 2.0 ** -133 * 1.5, 2.0 ** -133 * 2.5, 3.0e38, 3.4e38,
           -(2.0 ** 128) * (1 - 2 ** -9), (2.0 ** 128) * (1 - 2 ** -9) * (1 - 2 ** -20)]
    got = ref.f64_to_bf16_bits(np.array(xs))
    for x, b in zip(xs, got):
        assert int(b) == bf16_bits_exact(Fraction(x)), x


def test_bf16_special_values():
    got = ref.f64_to_bf16_bits(np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -2.0]))
    assert list(got[:4]) == [0x0000, 0x8000, 0x7F80, 0xFF80]
    assert got[4] & 0x7F80 == 0x7F80 and got[4] & 0x7F
    assert list(got[5:]) == [0x3F80, 0xC000]


def test_bf16_bits_roundtrip():
    bits = np.arange(2 ** 16, dtype=np.uint32).astype(np.uint16)
    vals = ref.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    assert np.array_equal(ref.f64_to_bf16_bits(vals[finite]), bits[finite])


@pytest.mark.parametrize("k", [-133, -126, -1, 0, 1, 127])
def test_bf16_powers_of_two(k):
    assert ref.bf16_bits_to_f64(ref.f64_to_bf16_bits(np.ldexp(1.0, k))) == np.ldexp(1.0, k)
