"""Packed byte layouts, written from their specification. TEST INFRASTRUCTURE ONLY.

A packed matrix is one contiguous buffer of sections; every section starts at
a multiple of 256 bytes. W is N x K (output rows x input columns), row-major
along K; quantization blocks/groups of 128 run along K.

Ternary (2 bits per weight, code 00 = 0, 01 = +1, 10 = -1):
  section 0 codes : N x K/16 little-endian uint32 words; word (n, k // 16) holds
                    the 16 codes of k0 .. k0+15. Within a word the low 16 bits
                    hold the even columns and the high 16 bits the odd columns:
                    column r = k % 16 sits at bit r if r is even and at bit
                    15 + r if r is odd (2 bits, bit 0 of the code first).
  section 1 scales: N x K/128 fp16 bit patterns.

INT4 (4-bit two's complement, values -7 .. 7):
  section 0 codes : N x K/8 uint32 words; column r = k % 8 sits at bit 2r if r
                    is even and at bit 14 + 2r if r is odd (4 bits each).
  section 1 scales: N x K/128 fp16 bit patterns.

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


def ternary_sizes(N: int, K: int):
    return [N * K // 4, N * (K // 128) * 2]


def int4_sizes(N: int, K: int):
    return [N * K // 2, N * (K // 128) * 2]


def ternary_bit_pos(k):
    r = k % 16
    return r if r % 2 == 0 else 15 + r


def int4_bit_pos(k):
    r = k % 8
    return 2 * r if r % 2 == 0 else 14 + 2 * r
