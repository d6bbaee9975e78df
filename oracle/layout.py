"""Packed byte layouts, written from their specification. TEST INFRASTRUCTURE ONLY.

A packed matrix is one contiguous buffer of sections; every section starts at
a multiple of 256 bytes. W is N x K (output rows x input columns), row-major
along K; quantization blocks/groups of 128 run along K.

Ternary (2 bits per weight, code 00 = 0, 01 = +1, 10 = -1) and INT4 (4-bit
two's complement, values -7 .. 7) share one arrangement:

  section 0 codes : row-group records. Rows are taken in groups of 16 (the
                    last group padded with all-zero rows), columns in steps of
                    1024 (8 blocks of 128; the last step may hold fewer). The
                    record of (group g, step s) holds the 16 rows' codes of
                    that step, row after row, each row's nbk blocks in column
                    order (nbk = min(8, K/128 - 8s)). Records follow in (g, s)
                    order, so group g starts at g * 16 * K * bits / 8 and
                    step s of it at s * 16 * 8 * block_bytes. A block is
                    8 (ternary) or 16 (INT4) little-endian uint32 words:
                    * ternary word of columns k0..k0+15: the low 16 bits hold
                      the even columns, the high 16 bits the odd ones; column
                      r = k % 16 sits at bit r (r even) or 15 + r (r odd),
                      2 bits each, code bit 0 first;
                    * INT4 word of columns k0..k0+7: column r = k % 8 at bit
                      2r (r even) or 14 + 2r (r odd), 4 bits each.
  section 1 scales: fp16 bit patterns in the same record order as the codes:
                    the record of (group g, step s) is 16 rows x 8 scales
                    (256 bytes; rows past N and blocks past K/128 hold 0), so
                    the scale of (row n, block b) is element
                    ((n // 16) * S + b // 8) * 128 + (n % 16) * 8 + b % 8,
                    with S = ceil(K / 1024) steps per row.

Ternary in the byte-lookup layout (the same codes and scales, arranged for a
matvec that reads one code byte per table lookup): rows go in NG = ceil(N/32)
groups of 32 (the last padded with zero codes and zero scales), KB = K/128.

  section 0 codes : NG * KB * 1024 bytes. Byte c of a row's block holds the
                    codes of columns 4c .. 4c+3 of the block, column 4c + i at
                    bits 2i, 2i+1. A row's 32 bytes of a block are rotated by
                    n % 32: the byte at position t is byte (t + n) % 32. The
                    1024-byte record of (block b, row group G) starts at
                    (b * NG + G) * 1024; position t of row n lies at
                    (t // 16) * 512 + (n % 32) * 16 + t % 16 inside it.
  section 1 scales: fp16 bits [KB][NG * 32]; (row n, block b) is element
                    b * NG * 32 + n.

INT4 in the byte-lookup layout (the same codes and scales as INT4, arranged for
a matvec that reads one code byte, a column pair, per table lookup): rows in
NG = ceil(N/32) groups of 32 (the last padded with zero codes and zero scales),
KB = K/128.

  section 0 codes : NG * KB * 2048 bytes. Byte p of a row's block holds the
                    codes of columns 2p (low nibble) and 2p + 1 (high nibble),
                    4-bit two's complement. A row's 64 bytes of a block are
                    read as two halves of 32, each rotated by n % 32: position
                    t < 32 holds byte (t + n) % 32, position t >= 32 holds byte
                    32 + (t - 32 + n) % 32. The 2048-byte record of (block b,
                    row group G) starts at (b * NG + G) * 2048; position t of
                    row n lies at (t // 16) * 512 + (n % 32) * 16 + t % 16.
  section 1 scales: fp16 bits [KB][NG * 32], as in the ternary lookup layout.

Cassandra split (see ``oracle.cassandra`` for the contents):
  0 bitmap    : N x K/32 uint32, bit (j % 32) of word j // 32 = kept(n, j)
  1 signmant  : N x (K/2)/8 uint32, nibble i (bits 4(i%8)..) = S<<3 | M>>4 of
                the i-th kept value of the row, column order
  2 expstream : unary exponent codes, LSB-first bits in uint32 words; each
                row starts on a 16-byte boundary, zero padded
  3 rowstart  : N + 1 uint32, first word of each row's stream (last = total)
  4 codebook  : 256 bytes, codebook[rank] = exponent field E
  5 pruned    : N x K/2 uint16, raw bf16 bits of the pruned values, column order
  6 mlo       : N x (K/2)/8 uint32, nibble i = M & 0xF of the i-th kept value
"""
from __future__ import annotations

import numpy as np

ALIGN = 256


def align(n: int, a: int = ALIGN) -> int:
    return (n + a - 1) // a * a


def sections(sizes):
    """Offsets of consecutive sections, each aligned to 256 bytes; returns (offsets, total)."""
    offs = []
    pos = 0
    for s in sizes:
        offs.append(pos)
        pos = align(pos + s)
    return offs, pos


ROW_GROUP = 16
STEP_BLOCKS = 8


def padded_rows(N: int) -> int:
    return (N + ROW_GROUP - 1) // ROW_GROUP * ROW_GROUP


def steps(K: int) -> int:
    """Steps of 1024 columns per row (the last one may hold fewer blocks)."""
    return (K // 128 + STEP_BLOCKS - 1) // STEP_BLOCKS


def scale_section_bytes(N: int, K: int) -> int:
    return padded_rows(N) // ROW_GROUP * steps(K) * ROW_GROUP * STEP_BLOCKS * 2


def ternary_sizes(N: int, K: int):
    return [padded_rows(N) * K // 4, scale_section_bytes(N, K)]


def int4_sizes(N: int, K: int):
    return [padded_rows(N) * K // 2, scale_section_bytes(N, K)]


def payload_bytes(N: int, K: int, bits: int) -> int:
    """Bytes of information in a block-128 matrix: the codes and one fp16 scale per block."""
    return N * K * bits // 8 + N * (K // 128) * 2


def scale_index(n: int, b: int, K: int) -> int:
    """Element index of the scale of (row n, block b) in section 1."""
    return ((n // ROW_GROUP) * steps(K) + b // STEP_BLOCKS) * (ROW_GROUP * STEP_BLOCKS) + \
        (n % ROW_GROUP) * STEP_BLOCKS + b % STEP_BLOCKS


def scale_indices(N: int, K: int):
    """scale_index for every (row, block) of an N x K matrix, as an [N][K/128] array."""
    n = np.arange(N)[:, None]
    b = np.arange(K // 128)[None, :]
    return scale_index(n, b, K)


def scale_records_from_rows(s16, K: int):
    """fp16 scale bits [N][K/128] -> section 1 (uint16, record order, zero padded)."""
    N = s16.shape[0]
    out = np.zeros(scale_section_bytes(N, K) // 2, dtype=np.uint16)
    out[scale_indices(N, K)] = s16
    return out


def rows_from_scale_records(flat, N: int, K: int):
    """Inverse of scale_records_from_rows."""
    return np.asarray(flat)[scale_indices(N, K)].astype(np.uint16)


def records_from_rows(words, block_words: int):
    """Row-major code words [N][K/cpw] -> the row-group record order of section 0."""
    N, W = words.shape
    KB = W // block_words
    Np = padded_rows(N)
    rows = np.zeros((Np, W), dtype=np.uint32)
    rows[:N] = words
    out = []
    for g in range(Np // ROW_GROUP):
        grp = rows[g * ROW_GROUP:(g + 1) * ROW_GROUP]
        for s in range(0, KB, STEP_BLOCKS):
            nbk = min(STEP_BLOCKS, KB - s)
            out.append(grp[:, s * block_words:(s + nbk) * block_words].ravel())
    return np.concatenate(out) if out else np.zeros(0, dtype=np.uint32)


def rows_from_records(flat, N: int, K: int, block_words: int, cols_per_word: int):
    """Inverse of records_from_rows: section 0 words -> row-major [N][K/cpw]."""
    KB = K // 128
    W = K // cols_per_word
    Np = padded_rows(N)
    rows = np.zeros((Np, W), dtype=np.uint32)
    pos = 0
    for g in range(Np // ROW_GROUP):
        for s in range(0, KB, STEP_BLOCKS):
            nbk = min(STEP_BLOCKS, KB - s)
            n = ROW_GROUP * nbk * block_words
            rows[g * ROW_GROUP:(g + 1) * ROW_GROUP, s * block_words:(s + nbk) * block_words] = \
                flat[pos:pos + n].reshape(ROW_GROUP, nbk * block_words)
            pos += n
    return rows[:N]


LUT_ROW_GROUP = 32


def lut_groups(N: int) -> int:
    return (N + LUT_ROW_GROUP - 1) // LUT_ROW_GROUP


def ternary_lut_sizes(N: int, K: int):
    NG, KB = lut_groups(N), K // 128
    return [NG * KB * 1024, KB * NG * LUT_ROW_GROUP * 2]


def lut_byte_offset(n: int, b: int, t: int, N: int) -> int:
    """Offset in section 0 of position t of (row n, block b)."""
    NG = lut_groups(N)
    return (b * NG + n // LUT_ROW_GROUP) * 1024 + (t // 16) * 512 + (n % LUT_ROW_GROUP) * 16 + t % 16


def lut_scale_index(n: int, b: int, N: int) -> int:
    return b * lut_groups(N) * LUT_ROW_GROUP + n


def int4_lut_sizes(N: int, K: int):
    NG, KB = lut_groups(N), K // 128
    return [NG * KB * 2048, KB * NG * LUT_ROW_GROUP * 2]


def lut4_byte_offset(n: int, b: int, t: int, N: int) -> int:
    """Offset in section 0 of position t (0..63) of (row n, block b), INT4 lookup layout."""
    NG = lut_groups(N)
    return (b * NG + n // LUT_ROW_GROUP) * 2048 + (t // 16) * 512 + (n % LUT_ROW_GROUP) * 16 + t % 16


def lut4_pair_at(n: int, t: int) -> int:
    """The column pair whose byte sits at position t of row n (two halves, each rotated by n % 32)."""
    half = t // 32
    return 32 * half + (t % 32 + n) % 32


def ternary_bit_pos(k):
    r = k % 16
    return r if r % 2 == 0 else 15 + r


def int4_bit_pos(k):
    r = k % 8
    return 2 * r if r % 2 == 0 else 14 + 2 * r
