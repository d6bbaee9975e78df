"""Symmetric group-128 absmax/7 INT4 quantizer and its packed form. TEST INFRASTRUCTURE ONLY.

Follows the group-wise step of "GPT-5.4 ..." section 3.2: per group of 128
weights, scales = max|w| / 7 and q = round(w / scales).clamp(-7, 7) stored as
int8. Readings:

* ``round`` is round-half-to-even (torch.round); the decision uses the
  unrounded float64 scale, the stored scale is its fp16 rounding;
* groups run along K (the input dimension) of the N x K matrix;
* an all-zero group has max|w| = 0: q = 0 and stored scale 0 (the page's
  0/0 is undefined);
* q is stored as a 4-bit two's-complement nibble; -8 is never produced.
"""
from __future__ import annotations

import numpy as np

from . import layout
from .numerics import f16_bits_to_f64, f64_to_f16_bits

GROUP = 128


def quantize(w: np.ndarray):
    """w float32 [N][K] -> (q int8 [N][K], s_star float64 [N][K/128], s16 uint16)."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % GROUP == 0
    g = w.astype(np.float64).reshape(N, K // GROUP, GROUP)
    s_star = np.abs(g).max(axis=2) / 7.0
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.rint(g / s_star[:, :, None])
    r = np.where(s_star[:, :, None] == 0.0, 0.0, r)
    q = np.clip(r, -7, 7).astype(np.int8)
    return q.reshape(N, K), s_star, f64_to_f16_bits(s_star)


def pack(q: np.ndarray, s16: np.ndarray) -> bytes:
    N, K = q.shape
    nib = (np.asarray(q).astype(np.int32) & 0xF).astype(np.uint32).reshape(N, K // 8, 8)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for r in range(8):
        words |= nib[:, :, r] << np.uint32(layout.int4_bit_pos(r))
    offs, total = layout.sections(layout.int4_sizes(N, K))
    buf = bytearray(total)
    rec = layout.records_from_rows(words, 16)
    buf[offs[0]:offs[0] + rec.nbytes] = rec.astype("<u4").tobytes()
    s = layout.scale_records_from_rows(np.asarray(s16, dtype=np.uint16), K).astype("<u2")
    buf[offs[1]:offs[1] + s.nbytes] = s.tobytes()
    return bytes(buf)


def unpack(buf: bytes, N: int, K: int):
    offs, total = layout.sections(layout.int4_sizes(N, K))
    assert len(buf) >= total
    flat = np.frombuffer(buf, dtype="<u4", count=layout.padded_rows(N) * K // 8, offset=offs[0])
    words = layout.rows_from_records(flat, N, K, 16, 8)
    q = np.empty((N, K // 8, 8), dtype=np.int8)
    for r in range(8):
        nib = ((words >> np.uint32(layout.int4_bit_pos(r))) & 0xF).astype(np.int32)
        q[:, :, r] = np.where(nib >= 8, nib - 16, nib)
    flat_s = np.frombuffer(buf, dtype="<u2", count=layout.scale_section_bytes(N, K) // 2, offset=offs[1])
    s16 = layout.rows_from_scale_records(flat_s, N, K)
    return q.reshape(N, K), s16.copy()


def pack_lut(q: np.ndarray, s16: np.ndarray) -> bytes:
    """Packed INT4 buffer in the byte-lookup layout (``oracle.layout``), by plain loops over
    rows, blocks and byte positions."""
    N, K = q.shape
    KB = K // GROUP
    nib = (np.asarray(q).astype(np.int32) & 0xF).reshape(N, KB, 64, 2)   # [row][block][pair][column]
    pair_bytes = nib[:, :, :, 0] | (nib[:, :, :, 1] << 4)
    offs, total = layout.sections(layout.int4_lut_sizes(N, K))
    buf = bytearray(total)
    for n in range(N):
        for b in range(KB):
            for t in range(64):
                buf[offs[0] + layout.lut4_byte_offset(n, b, t, N)] = int(pair_bytes[n, b, layout.lut4_pair_at(n, t)])
    s16 = np.asarray(s16, dtype=np.uint16)
    for n in range(N):
        for b in range(KB):
            pos = offs[1] + 2 * layout.lut_scale_index(n, b, N)
            buf[pos:pos + 2] = int(s16[n, b]).to_bytes(2, "little")
    return bytes(buf)


def unpack_lut(buf: bytes, N: int, K: int):
    """Inverse of ``pack_lut``: (q int8 [N][K], s16 uint16 [N][K/128])."""
    KB = K // GROUP
    offs, total = layout.sections(layout.int4_lut_sizes(N, K))
    assert len(buf) >= total
    raw = np.frombuffer(buf, dtype=np.uint8)
    q = np.zeros((N, K), dtype=np.int8)
    s16 = np.zeros((N, KB), dtype=np.uint16)
    for n in range(N):
        for b in range(KB):
            for t in range(64):
                byte = int(raw[offs[0] + layout.lut4_byte_offset(n, b, t, N)])
                p = layout.lut4_pair_at(n, t)
                for i, v in enumerate((byte & 0xF, byte >> 4)):
                    q[n, b * GROUP + 2 * p + i] = v - 16 if v >= 8 else v
            pos = offs[1] + 2 * layout.lut_scale_index(n, b, N)
            s16[n, b] = int.from_bytes(bytes(raw[pos:pos + 2]), "little")
    return q, s16


def dequant(q: np.ndarray, s16: np.ndarray) -> np.ndarray:
    N, K = q.shape
    s = f16_bits_to_f64(s16)
    return (q.reshape(N, K // GROUP, GROUP).astype(np.float64) * s[:, :, None]).reshape(N, K)
