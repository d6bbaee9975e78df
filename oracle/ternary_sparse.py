"""Flagged sparse ternary: block_ternary with all-zero tiles left out. TEST INFRASTRUCTURE ONLY.

Written from "Ternary Bonsai 2", sections 1.1, 1.3, 3.3, 3.4 and 5.5: blocks whose
weights are all zero carry a flag, their scale is fixed to 1 (no division by a zero
mean), and structured block-level sparsity with a sparse index brings the format
below 2 bits per parameter (about 1.78 on the page's 27B model).

Readings (the page gives no layout):
* quantization is ``oracle.ternary``'s block_ternary; a block whose codes are all
  zero stores the scale 1.0 (fp16 0x3C00) instead of fp16(1e-8) = 0;
* the sparse unit is a tile of 16 rows (one row group of the packed layout) x one
  block of 128 columns; a tile whose 16 x 128 codes are all zero (rows past N count
  as zero) is flagged in the group's tile bitmap and not stored;
* stored tiles of a group keep column order and are cut into records of up to 8
  tiles: a record is the 16 rows' code blocks of its tiles, row after row (the
  dense layout's record with its block list compacted).

Layout (sections 256-byte aligned):
  0 tilemap  : G x ceil(KB/32) uint32, bit (b % 32) of word b // 32 = tile (g, b) stored
  1 tilestart: G + 1 uint32, stored tiles before group g (last = T, all stored tiles)
  2 tileblock: T uint16, block index b of each stored tile, group by group
  3 codes    : group by group, records of 8 stored tiles; T * 16 * 8 words in all
  4 scales   : T x 16 fp16, the 16 rows' scales of each stored tile
with G = ceil(N / 16) groups and KB = K / 128 blocks per row.
"""
from __future__ import annotations

import numpy as np

from . import layout, ternary

SCALE_ONE = 0x3C00


def quantize(w: np.ndarray):
    """block_ternary codes and stored fp16 scales, all-zero blocks at scale 1.0."""
    q, s, s16 = ternary.quantize(w)
    N, K = q.shape
    zero_block = ~np.any(q.reshape(N, K // 128, 128) != 0, axis=2)
    s16 = np.where(zero_block, SCALE_ONE, s16).astype(np.uint16)
    return q, s16


def tile_stored(q: np.ndarray) -> np.ndarray:
    """bool [G][KB]: True where the 16-row x 128-column tile has a nonzero code."""
    N, K = q.shape
    G = layout.padded_rows(N) // 16
    qp = np.zeros((G * 16, K), dtype=q.dtype)
    qp[:N] = q
    return np.any(qp.reshape(G, 16, K // 128, 128) != 0, axis=(1, 3))


def sizes(N: int, K: int, T: int):
    G = layout.padded_rows(N) // 16
    KB = K // 128
    return [G * ((KB + 31) // 32) * 4, (G + 1) * 4, T * 2, T * 16 * 8 * 4, T * 16 * 2]


def pack(q: np.ndarray, s16: np.ndarray):
    """(buffer bytes, meta) of the flagged sparse layout."""
    N, K = q.shape
    KB = K // 128
    G = layout.padded_rows(N) // 16
    stored = tile_stored(q)
    T = int(stored.sum())
    # code words of every (row, block) as in the dense format: [Np][KB][8]
    c = ternary.codes_of(q).reshape(N, K // 16, 16)
    words = np.zeros((N, K // 16), dtype=np.uint32)
    for r in range(16):
        words |= c[:, :, r] << np.uint32(layout.ternary_bit_pos(r))
    wp = np.zeros((G * 16, KB, 8), dtype=np.uint32)
    wp[:N] = words.reshape(N, KB, 8)
    sp = np.zeros((G * 16, KB), dtype=np.uint16)
    sp[:N] = s16
    tilemap = np.zeros((G, (KB + 31) // 32), dtype=np.uint32)
    tilestart = np.zeros(G + 1, dtype=np.uint32)
    tileblock, codes, scales = [], [], []
    for g in range(G):
        blocks = np.flatnonzero(stored[g])
        for b in blocks:
            tilemap[g, b // 32] |= np.uint32(1) << np.uint32(b % 32)
        tilestart[g + 1] = tilestart[g] + len(blocks)
        tileblock.extend(blocks.tolist())
        rows = wp[g * 16:(g + 1) * 16]                    # [16][KB][8]
        for r0 in range(0, len(blocks), 8):
            sel = blocks[r0:r0 + 8]
            codes.append(rows[:, sel, :].reshape(-1))     # 16 rows, each its nbk tiles in order
        for b in blocks:
            scales.append(sp[g * 16:(g + 1) * 16, b])
    parts = [tilemap, tilestart, np.array(tileblock, dtype=np.uint16),
             np.concatenate(codes) if codes else np.zeros(0, np.uint32),
             np.concatenate(scales).astype(np.uint16) if scales else np.zeros(0, np.uint16)]
    raw = [np.ascontiguousarray(p).astype(p.dtype.newbyteorder("<")).tobytes() for p in parts]
    assert [len(r) for r in raw] == sizes(N, K, T)
    offs, total = layout.sections([len(r) for r in raw])
    buf = bytearray(total)
    for o, r in zip(offs, raw):
        buf[o:o + len(r)] = r
    return bytes(buf), dict(N=N, K=K, T=T, offsets=offs, sizes=[len(r) for r in raw], total=total, stored=stored)


def unpack(buf: bytes, meta):
    """Inverse of ``pack``: (q int8 [N][K], s16 [N][K/128]); left-out tiles give q = 0, scale 1.0."""
    N, K, T = meta["N"], meta["K"], meta["T"]
    KB = K // 128
    G = layout.padded_rows(N) // 16
    o = meta["offsets"]
    tilemap = np.frombuffer(buf, "<u4", G * ((KB + 31) // 32), o[0]).reshape(G, -1)
    tilestart = np.frombuffer(buf, "<u4", G + 1, o[1])
    tileblock = np.frombuffer(buf, "<u2", T, o[2])
    codes = np.frombuffer(buf, "<u4", T * 128, o[3])
    scales = np.frombuffer(buf, "<u2", T * 16, o[4]).reshape(T, 16)
    wp = np.zeros((G * 16, KB, 8), dtype=np.uint32)
    sp = np.full((G * 16, KB), SCALE_ONE, dtype=np.uint16)
    pos = 0
    for g in range(G):
        t0, t1 = int(tilestart[g]), int(tilestart[g + 1])
        blocks = tileblock[t0:t1].astype(np.int64)
        for b in blocks:
            assert (tilemap[g, b // 32] >> np.uint32(b % 32)) & 1
        for r0 in range(0, len(blocks), 8):
            sel = blocks[r0:r0 + 8]
            n = 16 * len(sel) * 8
            wp[g * 16:(g + 1) * 16, sel, :] = codes[pos:pos + n].reshape(16, len(sel), 8)
            pos += n
        for i, b in enumerate(blocks):
            sp[g * 16:(g + 1) * 16, b] = scales[t0 + i]
    words = wp[:N].reshape(N, K // 16)
    c = np.empty((N, K // 16, 16), dtype=np.uint32)
    for r in range(16):
        c[:, :, r] = (words >> np.uint32(layout.ternary_bit_pos(r))) & 3
    q = np.where(c == 1, 1, np.where(c == 2, -1, 0)).astype(np.int8).reshape(N, K)
    return q, sp[:N]


def bits_per_weight(N: int, K: int, T: int) -> float:
    return sum(sizes(N, K, T)) * 8 / (N * K)
