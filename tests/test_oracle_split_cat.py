"""Pins of the oracle's split + cat epilogue (a reading of a name the pages
give without semantics: blog analysis of sglang PR #39598, section 2,
``fused_gemm_afp4wfp4_split_cat`` and the 5-tuple input comment).

The reading: the GEMM output's N columns form H groups of s1 + s2; group h's
first s1 columns followed by z[m, h] form cat[m, h], its last s2 columns
split[m, h].  The pins: a small case worked out by hand, the inverse (y and z
rebuilt from the two outputs), and the degenerate groups (no split part, no
concatenated tensor, a single group).
"""

import numpy as np

from oracle import mxfp4_ref as ref


def test_hand_worked_example():
    # y row 0 = 0..11 as "bits", two groups of s1 = 2, s2 = 4; z row 0 = [[100], [101]]
    y = np.arange(12, dtype=np.uint16)[None, :]
    z = np.array([[[100], [101]]], dtype=np.uint16)
    cat, split = ref.split_cat(y, z, 2, 4)
    assert cat.tolist() == [[[0, 1, 100], [6, 7, 101]]]
    assert split.tolist() == [[[2, 3, 4, 5], [8, 9, 10, 11]]]


def test_inverse_rebuilds_y_and_z():
    g = np.random.default_rng(0)
    M, H, s1, s2, s3 = 5, 7, 16, 24, 40
    y = g.integers(0, 65536, size=(M, H * (s1 + s2)), dtype=np.uint16)
    z = g.integers(0, 65536, size=(M, H, s3), dtype=np.uint16)
    cat, split = ref.split_cat(y, z, s1, s2)
    rebuilt = np.concatenate([cat[:, :, :s1], split], axis=2).reshape(M, -1)
    assert np.array_equal(rebuilt, y)
    assert np.array_equal(cat[:, :, s1:], z)


def test_degenerate_groups():
    g = np.random.default_rng(1)
    y = g.integers(0, 65536, size=(3, 32), dtype=np.uint16)
    # no split part: cat = the whole group, then z
    z = g.integers(0, 65536, size=(3, 4, 8), dtype=np.uint16)
    cat, split = ref.split_cat(y, z, 8, 0)
    assert split.shape == (3, 4, 0)
    assert np.array_equal(cat[:, :, :8].reshape(3, 32), y)
    # no concatenated tensor: cat and split are the two column ranges of each group
    cat, split = ref.split_cat(y, np.zeros((3, 2, 0), np.uint16), 8, 8)
    assert np.array_equal(cat.reshape(3, 2, 8), y.reshape(3, 2, 16)[:, :, :8])
    assert np.array_equal(split, y.reshape(3, 2, 16)[:, :, 8:])
    # one group: an ordinary column split of y, then z appended to the first part
    z1 = g.integers(0, 65536, size=(3, 1, 16), dtype=np.uint16)
    cat, split = ref.split_cat(y, z1, 24, 8)
    assert np.array_equal(cat[:, 0], np.concatenate([y[:, :24], z1[:, 0]], axis=1))
    assert np.array_equal(split[:, 0], y[:, 24:])
