"""Block-128 absmean ternary quantizer and its packed form. TEST INFRASTRUCTURE ONLY.

Follows ``block_ternary(w, block_size=128, eps=1e-8)`` of "Ternary Bonsai 2",
section 1.2: per block of 128 consecutive weights along K,
scale = mean(|w|) + eps and q = clamp(round(w / scale), -1, 1). Readings where
the page is silent or garbled:

* the ``+`` before ``eps`` was lost in extraction; the scale is mean|w| + 1e-8;
* ``round`` is round-half-to-even (torch.round);
* the decision uses the unrounded float64 scale; the stored scale is that
  value rounded to fp16 (nearest even), which is what dequantization uses;
* mean|w| is the float64 sum over k = 0..127 in order, divided by 128;
* an all-zero block has scale 1e-8, q = 0 and a stored fp16 scale of 0
  (section 3.4 / 5.5 describe such blocks; no flag is stored in this format).
"""
from __future__ import annotations

import numpy as np

from . import layout
from .numerics import f16_bits_to_f64, f64_to_f16_bits

BLOCK = 128
EPS = 1e-8
CODE = {0: 0b00, 1: 0b01, -1: 0b10}


def quantize(w: np.ndarray):
    """w float32 [N][K] -> (q int8 [N][K], s_star float64 [N][K/128], s16 uint16 [N][K/128])."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % BLOCK == 0
    blocks = w.astype(np.float64).reshape(N, K // BLOCK, BLOCK)
    acc = np.zeros((N, K // BLOCK), dtype=np.float64)
    for k in range(BLOCK):                       # sum |w| in column order
        acc += np.abs(blocks[:, :, k])
    s_star = acc / BLOCK + EPS
    q = np.clip(np.rint(blocks / s_star[:, :, None]), -1, 1).astype(np.int8)
    return q.reshape(N, K), s_star, f64_to_f16_bits(s_star)


def codes_of(q: np.ndarray) -> np.ndarray:
    q = np.asarray(q)
    return np.where(q == 1, 1, np.where(q == -1, 2, 0)).astype(np.uint32)


def pack(q: np.ndarray, s16: np.ndarray) -> bytes:
    """Packed ternary buffer (layout in ``oracle.layout``)."""
    N, K = q.shape
    c = codes_of(q).reshape(N, K // 16, 16)
    words = np.zeros((N, K // 16), dtype=np.uint32)
    for r in range(16):
        words |= c[:, :, r] << np.uint32(layout.ternary_bit_pos(r))
    offs, total = layout.sections(layout.ternary_sizes(N, K))
    buf = bytearray(total)
    rec = layout.records_from_rows(words, 8)
    buf[offs[0]:offs[0] + rec.nbytes] = rec.astype("<u4").tobytes()
    s = layout.scale_records_from_rows(np.asarray(s16, dtype=np.uint16), K).astype("<u2")
    buf[offs[1]:offs[1] + s.nbytes] = s.tobytes()
    return bytes(buf)


def unpack(buf: bytes, N: int, K: int):
    """Inverse of ``pack``: (q int8 [N][K], s16 uint16 [N][K/128]). Code 11 is rejected."""
    offs, total = layout.sections(layout.ternary_sizes(N, K))
    assert len(buf) >= total
    flat = np.frombuffer(buf, dtype="<u4", count=layout.padded_rows(N) * K // 16, offset=offs[0])
    words = layout.rows_from_records(flat, N, K, 8, 16)
    c = np.empty((N, K // 16, 16), dtype=np.uint32)
    for r in range(16):
        c[:, :, r] = (words >> np.uint32(layout.ternary_bit_pos(r))) & 3
    if np.any(c == 3):
        raise ValueError("invalid ternary code 11")
    q = np.where(c == 1, 1, np.where(c == 2, -1, 0)).astype(np.int8).reshape(N, K)
    flat_s = np.frombuffer(buf, dtype="<u2", count=layout.scale_section_bytes(N, K) // 2, offset=offs[1])
    s16 = layout.rows_from_scale_records(flat_s, N, K)
    return q, s16.copy()


def pack_lut(q: np.ndarray, s16: np.ndarray) -> bytes:
    """Packed ternary buffer in the byte-lookup layout (``oracle.layout``), by plain loops
    over rows, blocks and byte positions."""
    N, K = q.shape
    KB = K // BLOCK
    c = codes_of(q).reshape(N, KB, 32, 4)              # [row][block][column group][column in group]
    group_bytes = np.zeros((N, KB, 32), dtype=np.uint32)
    for i in range(4):
        group_bytes |= c[:, :, :, i] << np.uint32(2 * i)
    offs, total = layout.sections(layout.ternary_lut_sizes(N, K))
    buf = bytearray(total)
    for n in range(N):
        for b in range(KB):
            for t in range(32):
                buf[offs[0] + layout.lut_byte_offset(n, b, t, N)] = int(group_bytes[n, b, (t + n) % 32])
    s16 = np.asarray(s16, dtype=np.uint16)
    for n in range(N):
        for b in range(KB):
            pos = offs[1] + 2 * layout.lut_scale_index(n, b, N)
            buf[pos:pos + 2] = int(s16[n, b]).to_bytes(2, "little")
    return bytes(buf)


def unpack_lut(buf: bytes, N: int, K: int):
    """Inverse of ``pack_lut``: (q int8 [N][K], s16 uint16 [N][K/128]). Code 11 is rejected."""
    KB = K // BLOCK
    offs, total = layout.sections(layout.ternary_lut_sizes(N, K))
    assert len(buf) >= total
    raw = np.frombuffer(buf, dtype=np.uint8)
    q = np.zeros((N, K), dtype=np.int8)
    s16 = np.zeros((N, KB), dtype=np.uint16)
    value = {0: 0, 1: 1, 2: -1}
    for n in range(N):
        for b in range(KB):
            for t in range(32):
                byte = int(raw[offs[0] + layout.lut_byte_offset(n, b, t, N)])
                grp = (t + n) % 32
                for i in range(4):
                    code = (byte >> (2 * i)) & 3
                    if code == 3:
                        raise ValueError("invalid ternary code 11")
                    q[n, b * BLOCK + 4 * grp + i] = value[code]
            pos = offs[1] + 2 * layout.lut_scale_index(n, b, N)
            s16[n, b] = int.from_bytes(bytes(raw[pos:pos + 2]), "little")
    return q, s16


def dequant(q: np.ndarray, s16: np.ndarray) -> np.ndarray:
    """w_hat = q * fp16 scale of its block, float64 [N][K]."""
    N, K = q.shape
    s = f16_bits_to_f64(s16)
    return (q.reshape(N, K // BLOCK, BLOCK).astype(np.float64) * s[:, :, None]).reshape(N, K)
