"""Online Cassandra encoder for the KV cache. TEST INFRASTRUCTURE ONLY.

Written from "Cassandra: ... self-speculative decoding" (cnblogs summary): the KV
cache is produced during decoding, so every new token's K/V values must be pruned,
truncated and unary-encoded on the spot before they are stored (section 3.5), and
the KV cache is pruned by per-token magnitude (section 3.2, step 1: keys have
channel outliers, so no activation norm enters the score).

Readings (the page gives no interface):
* a token's D values are one row; magnitude pruning keeps the D/2 largest |v| of
  the row, which is Cassandra-1's Wanda rule with every column norm equal to 1
  (equal magnitudes keep the lower index, NaN scores as +inf);
* the exponent ranking cannot be taken from the whole cache online, so the encoder
  is given a fixed codebook: all 256 exponent values in rank order (for instance a
  calibration ranking followed by the unseen exponents), rank r coded as r zeros
  then a one, as in Cassandra-1;
* each row's unary codes go into a fixed slot of ``slot_words`` 32-bit words
  (a multiple of 4), so rows can be encoded independently: rowstart[n] =
  n * slot_words, zero-filled after the codes; a row whose codes do not fit is an
  error (``fits`` is False for it here, the library records a status);
* everything else is Cassandra-1's layout (``oracle.cassandra``), so its draft and
  target decoders read the result unchanged.
"""
from __future__ import annotations

import numpy as np

from . import cassandra, layout


def magnitude_keep(W_bits: np.ndarray) -> np.ndarray:
    """bool [T][D]: the D/2 largest |v| of each row (ties: lower index; NaN as +inf)."""
    return cassandra.wanda_keep(W_bits, np.ones(W_bits.shape[1]))


def codebook_from(E_values: np.ndarray) -> np.ndarray:
    """All 256 exponents in rank order: those present in E_values by count (descending,
    equal counts smaller exponent first), then the absent ones in increasing order."""
    counts = np.bincount(np.asarray(E_values).ravel().astype(np.int64), minlength=256)
    present = sorted((e for e in range(256) if counts[e]), key=lambda e: (-counts[e], e))
    absent = [e for e in range(256) if not counts[e]]
    return np.array(present + absent, dtype=np.uint8)


def pack(W_bits: np.ndarray, codebook: np.ndarray, slot_words: int):
    """(buffer bytes, meta, fits [T] bool) in the Cassandra-1 layout with fixed stream slots."""
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    T, D = W_bits.shape
    assert D % 32 == 0 and slot_words % 4 == 0 and sorted(codebook.tolist()) == list(range(256))
    keep = magnitude_keep(W_bits)
    Sk, Ek, m_hi, m_lo, pruned = cassandra.split_values(W_bits, keep)
    rank_of = np.empty(256, dtype=np.int64)
    rank_of[codebook.astype(np.int64)] = np.arange(256)

    bitmap = np.zeros((T, D // 32), dtype=np.uint32)
    kb = keep.reshape(T, D // 32, 32).astype(np.uint32)
    for b in range(32):
        bitmap |= kb[:, :, b] << np.uint32(b)
    signmant = cassandra.nibbles_to_words((Sk << cassandra.M_HI_BITS) | m_hi)
    mlo = cassandra.nibbles_to_words(m_lo)
    stream = np.zeros((T, slot_words), dtype=np.uint32)
    fits = np.zeros(T, dtype=bool)
    for n in range(T):
        bits = cassandra.unary_bits(rank_of[Ek[n].astype(np.int64)])
        fits[n] = len(bits) <= slot_words * 32
        w = cassandra.bits_to_words(bits[: slot_words * 32])
        stream[n, : len(w)] = w
    rowstart = (np.arange(T + 1, dtype=np.uint32) * np.uint32(slot_words)).astype(np.uint32)

    parts = [bitmap, signmant, stream.reshape(-1), rowstart, codebook.astype(np.uint8), pruned.astype(np.uint16), mlo]
    raw = [np.ascontiguousarray(p).astype(p.dtype.newbyteorder("<")).tobytes() for p in parts]
    offs, total = layout.sections([len(r) for r in raw])
    buf = bytearray(total)
    for o, r in zip(offs, raw):
        buf[o:o + len(r)] = r
    meta = dict(N=T, K=D, offsets=offs, sizes=[len(r) for r in raw], total=total, n_symbols=256,
                codebook=codebook.copy(), keep=keep, stream_words=T * slot_words)
    return bytes(buf), meta, fits
