"""Pins for the fused RMSNorm -> MXFP4 oracle (CPU only).

Each check rests on something other than the oracle's own formula: a worked
example computed by hand, closed forms of RMSNorm (constant rows, scale
invariance, unit output RMS), bf16's round-half-to-even at exact ties, and
the placement of eps inside the root.
"""

import numpy as np
import pytest

from oracle import mxfp4_ref as ref
from oracle import rmsnorm_ref as rn

ONE = 0x3F80


def bits(vals):
    return ref.f64_to_bf16_bits(np.asarray(vals, dtype=np.float64))


def test_worked_example_by_hand():
    # x = [3, 4], gamma = 1, eps = 0:  mean square 12.5, so
    # y = [3, 4] / sqrt(12.5) = [0.84853, 1.13137].
    # bf16: 0.84853 / 2**-9 = 434.45 -> 434 * 2**-9 = 0.84765625 (0x3F59);
    #       1.13137 / 2**-7 = 144.82 -> 145 * 2**-7 = 1.1328125 (0x3F91).
    # quantization: amax 1.1328 -> floor(log2) = 0 -> E = -2, scale byte 125;
    # y / 0.25 = [3.39, 4.53] -> E2M1 3 (code 5) and 4 (code 6) -> byte 0x65.
    out = rn.rmsnorm_quant(np.array([[0x4040, 0x4080]], np.uint16), np.array([ONE, ONE], np.uint16), 0.0)
    assert out["y"].tolist() == [[0x3F59, 0x3F91]]
    assert out["scales"].tolist() == [[125]]
    assert out["codes"].tolist() == [[0x65]]


@pytest.mark.parametrize("c", [0.375, -3.0, 1e-20, 6e30])
def test_constant_row_gives_gamma(c):
    # h_i = c for all i: mean square c**2, so y_i = sign(c) * gamma_i exactly.
    K = 96
    gamma = bits(np.linspace(-2.0, 5.0, K))
    x = np.tile(bits([c]), (1, K))
    y = rn.rmsnorm_quant(x, gamma, 0.0)["y"]
    want = gamma if c > 0 else gamma ^ np.uint16(0x8000)
    assert np.array_equal(y[0], want)


def test_scale_invariance_without_eps():
    g = np.random.default_rng(0)
    x = bits(g.standard_normal((4, 160)))
    gamma = bits(g.uniform(0.5, 1.5, 160))
    base = rn.rmsnorm_quant(x, gamma, 0.0)
    for k in (-20, 7):
        scaled = bits(ref.bf16_bits_to_f64(x) * 2.0 ** k)     # exact: a power of two
        again = rn.rmsnorm_quant(scaled, gamma, 0.0)
        assert np.array_equal(again["y"], base["y"])
        assert np.array_equal(again["codes"], base["codes"]) and np.array_equal(again["scales"], base["scales"])


def test_unit_output_rms():
    g = np.random.default_rng(1)
    x = bits(g.standard_normal((3, 250)) * 7.0)
    y = rn.rmsnorm_quant(x, np.full(250, ONE, np.uint16), 0.0)["y_exact"]
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=0, atol=1e-12)


def test_eps_is_inside_the_root():
    # all ones, eps = 3: 1 / sqrt(1 + 3) = 0.5 (eps outside the root, or added
    # to the RMS instead, would give 0.25).
    y = rn.rmsnorm_quant(np.full((1, 32), ONE, np.uint16), np.full(32, ONE, np.uint16), 3.0)["y_exact"]
    assert np.all(y == 0.5)


def test_mean_is_over_k_not_the_padded_block():
    # K = 34 (two scale blocks, the second padded): all ones -> y = 1 exactly.
    y = rn.rmsnorm_quant(np.full((1, 34), ONE, np.uint16), np.full(34, ONE, np.uint16), 0.0)["y"]
    assert np.all(y == ONE)


def test_zero_row_and_nonfinite_rows():
    K = 64
    gamma = np.full(K, ONE, np.uint16)
    zero = rn.rmsnorm_quant(np.zeros((1, K), np.uint16), gamma, 1e-6)
    assert np.all(zero["y"] == 0) and np.all(zero["codes"] == 0) and np.all(zero["scales"] == 0)
    x = np.tile(bits([1.0]), (2, K))
    x[0, 5] = 0x7FC0        # NaN: the whole row becomes NaN
    x[1, 40] = 0x7F80       # Inf: that element becomes NaN (Inf / Inf), the others 0
    out = rn.rmsnorm_quant(x, gamma, 1e-6)
    assert np.all(out["scales"][0] == 0xFF) and np.all(out["codes"][0] == 0)
    assert out["scales"][1].tolist() == [0, 0xFF]
    assert np.all(ref.bf16_bits_to_f64(out["y"][1, :32]) == 0.0)


def test_residual_add_rounds_ties_to_even():
    # 1 + 2**-8 is halfway between bf16 1.0 (even) and 1.0078125: -> 1.0;
    # 1.0078125 + 2**-8 is halfway between 0x3F81 (odd) and 0x3F82: -> 0x3F82.
    x = np.array([[0x3F80, 0x3F81]], np.uint16)
    r = np.array([[0x3B80, 0x3B80]], np.uint16)
    assert rn.add_residual(x, r).tolist() == [[0x3F80, 0x3F82]]


def test_residual_then_norm_is_norm_of_the_sum():
    g = np.random.default_rng(2)
    x, res = bits(g.standard_normal((5, 96))), bits(g.standard_normal((5, 96)))
    gamma = bits(g.uniform(0.5, 1.5, 96))
    fused = rn.rmsnorm_quant(x, gamma, 1e-5, res_bits=res)
    assert np.array_equal(fused["h"], rn.add_residual(x, res))
    plain = rn.rmsnorm_quant(fused["h"], gamma, 1e-5)
    for k in ("y", "codes", "scales"):
        assert np.array_equal(fused[k], plain[k])
