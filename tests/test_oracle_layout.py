"""Pins of the oracle's packed tile layout (CPU only).

The oracle states the layout with vectorised index arithmetic.  Here it is
checked to be a bijection onto the packed buffer, against an independent
restatement (the 128-byte swizzle as an XOR of address bits, the scale atom
as a [32][4][4] array), for padding values, and for exact inversion.  The
pages' own AITER scale permutation (sglang PR #39598 blog analysis, sections
2 and 3: ``_swizzle_asm_fp4_scale`` and its CPU unit test on an arange) is
also checked to be a bijection, as a sanity check of the test pattern.
"""

import numpy as np
import pytest

from oracle import tile_layout as tl


@pytest.mark.parametrize("R,K", [(1, 32), (128, 256), (130, 5152), (300, 544), (1000, 5152)])
def test_offsets_are_bijections(R, K):
    co = tl.code_offsets(R, K).ravel()
    assert np.array_equal(np.sort(co), np.arange(tl.code_bytes(R, K)))
    so = tl.scale_offsets(R, K).ravel()
    assert np.array_equal(np.sort(so), np.arange(tl.scale_bytes(R, K)))


def expected_pack_by_address_bits(codes, scales, K):
    """Independent restatement: copy rows tile by tile, then XOR address bits."""
    R = codes.shape[0]
    Rp, Kp = tl.padded_dims(R, K)
    KT = Kp // 256
    cpad = np.zeros((Rp, Kp // 2), np.uint8)
    cpad[:R, :codes.shape[1]] = codes
    spad = np.full((Rp, Kp // 32), 0x7F, np.uint8)
    spad[:R, :scales.shape[1]] = scales
    out = []
    for rt in range(Rp // 128):
        for kt in range(KT):
            tile = cpad[rt * 128:(rt + 1) * 128, kt * 128:(kt + 1) * 128].ravel()
            sw = np.empty_like(tile)
            for o in range(16384):
                sw[o ^ (((o >> 7) & 7) << 4)] = tile[o]
            out.append(sw)
    for rt in range(Rp // 128):
        for g in range(Kp // 128):
            atom = np.empty((32, 4, 4), np.uint8)
            for i in range(128):
                for b in range(4):
                    atom[i % 32, i // 32, b] = spad[rt * 128 + i, g * 4 + b]
            out.append(atom.ravel())
    return np.concatenate(out)


@pytest.mark.parametrize("R,K", [(3, 64), (130, 544)])
def test_pack_matches_address_bit_restatement(R, K):
    g = np.random.default_rng(R + K)
    codes = g.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = g.integers(0, 256, size=(R, -(-K // 32)), dtype=np.uint8)
    assert np.array_equal(tl.pack(codes, scales, K), expected_pack_by_address_bits(codes, scales, K))


@pytest.mark.parametrize("R,K", [(1, 32), (17, 5152), (1000, 5152), (128, 5120)])
def test_unpack_inverts_pack_and_padding_values(R, K):
    g = np.random.default_rng(R * 7 + K)
    codes = g.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = g.integers(0, 255, size=(R, -(-K // 32)), dtype=np.uint8)
    packed = tl.pack(codes, scales, K)
    assert packed.size == tl.packed_bytes(R, K)
    c, s = tl.unpack(packed, R, K)
    assert np.array_equal(c[:R, :K // 2], codes)
    assert np.array_equal(s[:R, :scales.shape[1]], scales)
    assert np.all(c[R:] == 0) and np.all(c[:, K // 2:] == 0)
    assert np.all(s[R:] == 0x7F) and np.all(s[:, scales.shape[1]:] == 0x7F)


def test_batched_pack_concatenates():
    g = np.random.default_rng(1)
    codes = g.integers(0, 256, size=(3, 5, 32), dtype=np.uint8)
    scales = g.integers(0, 255, size=(3, 5, 2), dtype=np.uint8)
    p = tl.pack_batched(codes, scales, 64)
    per = tl.packed_bytes(5, 64)
    for b in range(3):
        assert np.array_equal(p[b * per:(b + 1) * per], tl.pack(codes[b], scales[b], 64))


def aiter_scale_order(scale):
    """The pages' tile order for a (rows, cols) scale tensor, rows % 32 == cols % 8 == 0."""
    rows, cols = scale.shape
    return (scale.reshape(rows // 32, 2, 16, cols // 8, 2, 4, 1)
            .transpose(0, 3, 5, 2, 4, 1, 6).reshape(rows, cols))


@pytest.mark.parametrize("rows,cols", [(32, 8), (64, 16), (96, 24)])
def test_page_aiter_permutation_is_bijection(rows, cols):
    a = np.arange(rows * cols).reshape(rows, cols)
    p = aiter_scale_order(a)
    assert np.array_equal(np.sort(p.ravel()), np.arange(rows * cols))
    # undoing the transpose restores the input
    back = (p.reshape(rows // 32, cols // 8, 4, 16, 2, 2, 1)
            .transpose(0, 5, 3, 1, 4, 2, 6).reshape(rows, cols))
    assert np.array_equal(back, a)


# ------------------------------------------------------------ weight layout
@pytest.mark.parametrize("R,K", [(1, 32), (256, 256), (300, 544), (1000, 5152), (130, 5120)])
def test_weight_offsets_partition_the_buffer(R, K):
    co = tl.weight_code_offsets(R, K).ravel()
    so = tl.weight_scale_offsets(R, K).ravel()
    both = np.concatenate([co, so])
    assert np.array_equal(np.sort(both), np.arange(tl.weight_packed_bytes(R, K)))
    Np, Kp = tl.weight_padded_dims(R, K)
    assert tl.weight_packed_bytes(R, K) == Np * Kp // 2 + Np * Kp // 32


def expected_weight_pack_by_blocks(codes, scales, K):
    """Independent restatement: per (row pair, k-tile) concatenate the two
    address-bit-swizzled code tiles and the four scale atoms."""
    R = codes.shape[0]
    Np, Kp = tl.weight_padded_dims(R, K)
    KT = Kp // 256
    cpad = np.zeros((Np, Kp // 2), np.uint8)
    cpad[:R, :codes.shape[1]] = codes
    spad = np.full((Np, Kp // 32), 0x7F, np.uint8)
    spad[:R, :scales.shape[1]] = scales
    out = []
    for p in range(Np // 256):
        for kt in range(KT):
            for h in range(2):
                r0 = p * 256 + h * 128
                tile = cpad[r0:r0 + 128, kt * 128:(kt + 1) * 128].ravel()
                sw = np.empty_like(tile)
                for o in range(16384):
                    sw[o ^ (((o >> 7) & 7) << 4)] = tile[o]
                out.append(sw)
            for h in range(2):
                r0 = p * 256 + h * 128
                for gq in range(2):
                    atom = np.empty((32, 4, 4), np.uint8)
                    for i in range(128):
                        for b in range(4):
                            atom[i % 32, i // 32, b] = spad[r0 + i, kt * 8 + gq * 4 + b]
                    out.append(atom.ravel())
    return np.concatenate(out)


@pytest.mark.parametrize("R,K", [(3, 64), (260, 544)])
def test_weight_pack_matches_block_restatement(R, K):
    g = np.random.default_rng(R * 3 + K)
    codes = g.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = g.integers(0, 256, size=(R, -(-K // 32)), dtype=np.uint8)
    assert np.array_equal(tl.pack_weights(codes, scales, K), expected_weight_pack_by_blocks(codes, scales, K))


@pytest.mark.parametrize("R,K", [(1, 32), (17, 5152), (1000, 5152), (256, 5120)])
def test_weight_unpack_inverts_pack_and_padding_values(R, K):
    g = np.random.default_rng(R * 11 + K)
    codes = g.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = g.integers(0, 255, size=(R, -(-K // 32)), dtype=np.uint8)
    packed = tl.pack_weights(codes, scales, K)
    c, s = tl.unpack_weights(packed, R, K)
    assert np.array_equal(c[:R, :K // 2], codes)
    assert np.array_equal(s[:R, :scales.shape[1]], scales)
    assert np.all(c[R:] == 0) and np.all(c[:, K // 2:] == 0)
    assert np.all(s[R:] == 0x7F) and np.all(s[:, scales.shape[1]:] == 0x7F)


def test_weight_block_holds_whole_tiles_and_atoms():
    """Rows 0..255 of k-tile 0 fill bytes [0, 34816) of the buffer: both code
    tiles first, the four scale atoms after them."""
    R, K = 512, 512
    co = tl.weight_code_offsets(R, K)
    so = tl.weight_scale_offsets(R, K)
    assert co[:256, :128].min() == 0 and co[:256, :128].max() == 32767
    assert so[:256, :8].min() == 32768 and so[:256, :8].max() == 34815
    assert co[256:, :128].min() == 2 * 34816          # pair 1 starts after pair 0's two k-tiles
