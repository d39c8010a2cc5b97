"""Property pins of the oracle's per-1x32 quantizer (CPU only), over blocks
drawn by hypothesis from the bf16 values: invariants any correct
round-to-nearest block quantizer has, independent of how the oracle computes
it.

* order: within a block (one shared scale) the dequantized values are a
  non-decreasing function of the inputs;
* sign symmetry: negating a block keeps its scale and flips every code's sign
  bit (a value that rounds to zero included: -0 encodes as 0x8);
* scale equivariance: multiplying a block by 2**j (no element leaving the
  normal bf16 range, the scale staying clear of the E8M0 clamp) adds j to the
  scale byte and leaves the codes unchanged;
* error bound: an element is off by at most half a grid step of its binade
  times the scale, unless it saturates at 6 * scale.
"""

import numpy as np
import pytest

from oracle import mxfp4_ref as ref

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings


def _bf16_finite(bits):
    return (bits & 0x7F80) != 0x7F80


block = st.lists(st.integers(0, 0xFFFF).filter(_bf16_finite), min_size=32, max_size=32)


def quantize(bits):
    x = ref.bf16_bits_to_f64(np.asarray(bits, dtype=np.uint16))[None, :]
    c, s = ref.quantize_mxfp4(x)
    return x[0], ref.unpack_codes(c, 32)[0].astype(np.int64), int(s[0, 0])


def deq(codes, sbyte):
    return ref.e2m1_decode(codes) * ref.e8m0_decode(np.array([sbyte]))[0]


@settings(max_examples=400, deadline=None)
@given(block)
def test_dequantized_order_follows_input_order(bits):
    x, codes, s = quantize(bits)
    d = deq(codes, s)
    order = np.argsort(x, kind="stable")
    assert np.all(np.diff(d[order]) >= 0)


@settings(max_examples=400, deadline=None)
@given(block)
def test_negation_flips_sign_bits_only(bits):
    neg = [b ^ 0x8000 for b in bits]
    _, c1, s1 = quantize(bits)
    _, c2, s2 = quantize(neg)
    assert s1 == s2
    assert np.array_equal(c1 ^ 0x8, c2)


def _mid_bits(t):
    sign, exp, man = t
    return (sign << 15) | (exp << 7) | man


# normal bf16 values with biased exponents 40..200: scaled by 2**j, |j| <= 20,
# they stay normal and the block scale (amax exponent - 2) stays off the clamp
mid_block = st.lists(st.tuples(st.integers(0, 1), st.integers(40, 200), st.integers(0, 127)).map(_mid_bits),
                     min_size=32, max_size=32)


@settings(max_examples=300, deadline=None)
@given(mid_block, st.integers(-20, 20))
def test_power_of_two_scaling_shifts_only_the_scale(bits, j):
    _, c1, s1 = quantize(bits)
    scaled = [(b & 0x807F) | ((((b >> 7) & 0xFF) + j) << 7) for b in bits]
    _, c2, s2 = quantize(scaled)
    assert s2 == s1 + j
    assert np.array_equal(c1, c2)


@settings(max_examples=400, deadline=None)
@given(block)
def test_error_within_half_a_grid_step_or_saturated(bits):
    x, codes, s = quantize(bits)
    scale = ref.e8m0_decode(np.array([s]))[0]
    d = deq(codes, s)
    q = np.abs(x) / scale
    # grid step of the E2M1 binade holding |x| / scale: 0.5 below 2, 1 in [2, 4), 2 from 4
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    sat = q > 6
    assert np.all(np.abs(d - x)[~sat] <= 0.5 * step[~sat] * scale)
    assert np.all(np.abs(d[sat]) == 6 * scale)
