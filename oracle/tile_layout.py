"""Plain statement of the packed "MMA tile" layout, for checking byte-exactly.

TEST INFRASTRUCTURE ONLY (see ``oracle/mxfp4_ref.py``).  This restates, with
numpy index arithmetic and nothing shared with the CUDA sources, the layout
that the library's one-time weight repack and its MMA-layout activation
quantizer write.  The pages' own repack is the AITER tile order for gfx950
(sglang PR #39598 blog analysis, section 2, ``_swizzle_asm_fp4_scale`` and
``shuffle_weight``); this layout is its Blackwell counterpart and is defined
by this library, not by the pages.

A matrix of R rows and K 4-bit elements (codes packed two per byte, scales one
per 32 elements) is padded to Rp = ceil(R/128)*128 rows and Kp = ceil(K/256)*256
elements.  Padding codes are 0, padding scales 0x7F (E8M0 1.0: the pages pad
with 1.0 because 0xFF would be NaN, blog analysis, section 2,
``_shuffle_asm_fp4_act_scale``).

Codes region, Rp*Kp/2 bytes: tiles of 128 rows x 128 bytes (256 elements),
tile (rt, kt) at byte ((rt * Kp/256) + kt) * 16384.  Inside a tile, byte j of
row i sits at i*128 + ((j//16) XOR (i % 8))*16 + j%16: the 128-byte swizzle of
the K-major shared-memory operand layout.

Scales region, Rp*Kp/32 bytes, right after the codes: atoms of 128 rows x 4
blocks (512 bytes), atom (rt, g) at ((rt * Kp/128) + g) * 512 for block group
g = block // 4; inside an atom the scale of row i, block b sits at
16*(i % 32) + 4*(i // 32) + b % 4.

A batch of matrices is stored one after another, each taking
``packed_bytes(R, K)`` bytes.

That is the layout of MMA-layout ACTIVATIONS (separate codes and scales
buffers).  Packed WEIGHTS use the same tiles and atoms grouped by pairs of
row tiles: rows are padded to Np = ceil(R/256)*256, and for each pair p (rows
256p..256p+255) and k-tile kt there is one contiguous block of 34816 bytes at
(p * Kp/256 + kt) * 34816 holding

    [code tile of rows 256p..+127 | code tile of rows 256p+128..+255 |
     2 scale atoms of the first 128 rows | 2 scale atoms of the second 128 rows]

(16384 + 16384 + 1024 + 1024 bytes; the atom of block group g, g = 0, 1 for
blocks 8kt..8kt+3 and 8kt+4..8kt+7, at 512*g inside each 1024).  Inside a
tile and an atom the byte positions are those above.  A batch of weight
matrices is stored one after another, ``weight_packed_bytes(R, K)`` each.
"""

from __future__ import annotations

import numpy as np

ROW_TILE = 128
K_TILE = 256            # elements per tile along K (128 bytes of codes)
SCALE_PAD = 0x7F
PAIR_ROWS = 256         # rows of one weight block
BLOCK_BYTES = 2 * 16384 + 2 * 1024


def padded_dims(R: int, K: int) -> tuple[int, int]:
    return -(-R // ROW_TILE) * ROW_TILE, -(-K // K_TILE) * K_TILE


def code_bytes(R: int, K: int) -> int:
    Rp, Kp = padded_dims(R, K)
    return Rp * Kp // 2


def scale_bytes(R: int, K: int) -> int:
    Rp, Kp = padded_dims(R, K)
    return Rp * Kp // 32


def packed_bytes(R: int, K: int) -> int:
    return code_bytes(R, K) + scale_bytes(R, K)


def code_offsets(R: int, K: int) -> np.ndarray:
    """Destination byte offset of packed code byte (r, j), j < Kp/2, all padded rows."""
    Rp, Kp = padded_dims(R, K)
    r = np.arange(Rp)[:, None]
    j = np.arange(Kp // 2)[None, :]
    rt, i = r // ROW_TILE, r % ROW_TILE
    kt, jj = j // 128, j % 128
    tile = rt * (Kp // K_TILE) + kt
    return tile * 16384 + i * 128 + (((jj // 16) ^ (i % 8)) * 16) + jj % 16


def scale_offsets(R: int, K: int) -> np.ndarray:
    """Offset (inside the scales region) of the scale of row r, block b."""
    Rp, Kp = padded_dims(R, K)
    r = np.arange(Rp)[:, None]
    b = np.arange(Kp // 32)[None, :]
    rt, i = r // ROW_TILE, r % ROW_TILE
    atom = rt * (Kp // 128) + b // 4
    return atom * 512 + 16 * (i % 32) + 4 * (i // 32) + b % 4


def pack(codes, scales, K: int) -> np.ndarray:
    """[R, K//2] codes + [R, ceil(K/32)] scales -> packed bytes (uint8 vector)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    R = codes.shape[0]
    Rp, Kp = padded_dims(R, K)
    cpad = np.zeros((Rp, Kp // 2), dtype=np.uint8)
    cpad[:R, : codes.shape[1]] = codes
    spad = np.full((Rp, Kp // 32), SCALE_PAD, dtype=np.uint8)
    spad[:R, : scales.shape[1]] = scales
    out = np.empty(packed_bytes(R, K), dtype=np.uint8)
    cb = code_bytes(R, K)
    out[code_offsets(R, K).ravel()] = cpad.ravel()
    out[cb + scale_offsets(R, K).ravel()] = spad.ravel()
    return out


def pack_batched(codes, scales, K: int) -> np.ndarray:
    """[B, R, K//2] + [B, R, ceil(K/32)] -> concatenated packed matrices."""
    return np.concatenate([pack(codes[b], scales[b], K) for b in range(codes.shape[0])])


def unpack(packed, R: int, K: int) -> tuple[np.ndarray, np.ndarray]:
    """Inverse of ``pack``: returns the padded [Rp, Kp/2] codes and [Rp, Kp/32] scales."""
    packed = np.asarray(packed, dtype=np.uint8)
    cb = code_bytes(R, K)
    codes = packed[code_offsets(R, K)]
    scales = packed[cb + scale_offsets(R, K)]
    return codes, scales


# ---------------------------------------------------------------- weights
def weight_padded_dims(R: int, K: int) -> tuple[int, int]:
    return -(-R // PAIR_ROWS) * PAIR_ROWS, -(-K // K_TILE) * K_TILE


def weight_packed_bytes(R: int, K: int) -> int:
    Np, Kp = weight_padded_dims(R, K)
    return (Np // PAIR_ROWS) * (Kp // K_TILE) * BLOCK_BYTES


def weight_code_offsets(R: int, K: int) -> np.ndarray:
    """Byte offset of packed weight code byte (r, j), j < Kp/2, all padded rows."""
    Np, Kp = weight_padded_dims(R, K)
    r = np.arange(Np)[:, None]
    j = np.arange(Kp // 2)[None, :]
    p, h, i = r // PAIR_ROWS, (r % PAIR_ROWS) // ROW_TILE, r % ROW_TILE
    kt, jj = j // 128, j % 128
    block = p * (Kp // K_TILE) + kt
    return block * BLOCK_BYTES + h * 16384 + i * 128 + (((jj // 16) ^ (i % 8)) * 16) + jj % 16


def weight_scale_offsets(R: int, K: int) -> np.ndarray:
    """Byte offset of the packed weight scale of row r, block b (same buffer as the codes)."""
    Np, Kp = weight_padded_dims(R, K)
    r = np.arange(Np)[:, None]
    b = np.arange(Kp // 32)[None, :]
    p, h, i = r // PAIR_ROWS, (r % PAIR_ROWS) // ROW_TILE, r % ROW_TILE
    kt, bb = b // 8, b % 8
    block = p * (Kp // K_TILE) + kt
    return (block * BLOCK_BYTES + 2 * 16384 + h * 1024 + (bb // 4) * 512
            + 16 * (i % 32) + 4 * (i // 32) + bb % 4)


def pack_weights(codes, scales, K: int) -> np.ndarray:
    """[R, K//2] codes + [R, ceil(K/32)] scales -> packed weight bytes (uint8 vector)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    R = codes.shape[0]
    Np, Kp = weight_padded_dims(R, K)
    cpad = np.zeros((Np, Kp // 2), dtype=np.uint8)
    cpad[:R, : codes.shape[1]] = codes
    spad = np.full((Np, Kp // 32), SCALE_PAD, dtype=np.uint8)
    spad[:R, : scales.shape[1]] = scales
    out = np.empty(weight_packed_bytes(R, K), dtype=np.uint8)
    out[weight_code_offsets(R, K).ravel()] = cpad.ravel()
    out[weight_scale_offsets(R, K).ravel()] = spad.ravel()
    return out


def pack_weights_batched(codes, scales, K: int) -> np.ndarray:
    """[B, R, K//2] + [B, R, ceil(K/32)] -> concatenated packed weight matrices."""
    return np.concatenate([pack_weights(codes[b], scales[b], K) for b in range(codes.shape[0])])


def unpack_weights(packed, R: int, K: int) -> tuple[np.ndarray, np.ndarray]:
    """Inverse of ``pack_weights``: the padded [Np, Kp/2] codes and [Np, Kp/32] scales."""
    packed = np.asarray(packed, dtype=np.uint8)
    return packed[weight_code_offsets(R, K)], packed[weight_scale_offsets(R, K)]
