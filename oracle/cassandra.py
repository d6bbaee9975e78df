"""Cassandra lossless bf16 split: speculation + verification data. TEST INFRASTRUCTURE ONLY.

Written from "Cassandra: ... self-speculative decoding" (cnblogs summary),
sections 3.1-3.3, in the order the page gives the offline transform:

1. value pruning (3.2, step 1): each weight gets the Wanda score
   |w| * ||X[:, j]||_2 over calibration activations X; the highest-scoring half
   of every output row is kept (speculation data), the rest is pruned into the
   verification data, and a bitmap records which were kept;
2. mantissa truncation (3.2, step 2): of a kept value's 7 mantissa bits the
   high 3 go to the speculation data, the low 4 to the verification data;
3. exponent compression (3.3, Cassandra-1): exponents are ranked by frequency;
   rank r is written as r zeros followed by a one (most frequent = "1").

Draft path (3.2, figure b): speculation data only; pruned positions read as
zero, truncated mantissa bits as zero. Target path (figure c): both streams
give back every original bit.

Readings where the page is silent:
* the column norm is the float64 sum over calibration rows in order, then sqrt;
* the score is |w| * c_j in float64; ties keep the lower column; a NaN weight
  scores +inf (kept); exactly K/2 values are kept per row ("top 50 %");
* frequencies are counted over all kept values of the tensor; equal counts
  rank the smaller exponent first; exponents that never occur get no rank;
* the high/low mantissa split is 3/4 bits; the draft fills the low bits with
  zeros (truncation, not rounding); pruned draft values are +0;
* stream layout (``oracle.layout``): kept values in column order, bits
  LSB-first in 32-bit words, each row's unary stream 16-byte aligned.
"""
from __future__ import annotations

import numpy as np

from . import layout
from .numerics import bf16_bits_to_f64, bf16_fields

M_HI_BITS = 3
M_LO_BITS = 4


def column_norms(X_bits: np.ndarray) -> np.ndarray:
    """c_j = sqrt(sum_r X[r][j]^2), float64, rows summed in order."""
    X = bf16_bits_to_f64(X_bits)
    acc = np.zeros(X.shape[1], dtype=np.float64)
    for r in range(X.shape[0]):
        acc += X[r] * X[r]
    return np.sqrt(acc)


def wanda_keep(W_bits: np.ndarray, c: np.ndarray) -> np.ndarray:
    """bool [N][K]: True where the value is kept (top K/2 of |w| * c_j per row)."""
    N, K = W_bits.shape
    w = bf16_bits_to_f64(W_bits)
    score = np.abs(w) * c[None, :]
    score = np.where(np.isnan(score), np.inf, score)
    cols = np.broadcast_to(np.arange(K), (N, K))
    order = np.lexsort((cols, -score), axis=1)     # score descending, then column ascending
    keep = np.zeros((N, K), dtype=bool)
    np.put_along_axis(keep, order[:, : K // 2], True, axis=1)
    return keep


def split_values(W_bits: np.ndarray, keep: np.ndarray):
    """Per-row column-order lists: kept (S, E, m_hi, m_lo) and pruned raw bits, each [N][K/2]."""
    N, K = W_bits.shape
    S, E, M = bf16_fields(W_bits)
    kept_cols = np.nonzero(keep)[1].reshape(N, K // 2)    # row-major order = column order per row
    pruned_cols = np.nonzero(~keep)[1].reshape(N, K // 2)
    take = lambda a, cols: np.take_along_axis(a, cols, axis=1)
    Sk, Ek, Mk = take(S, kept_cols), take(E, kept_cols), take(M, kept_cols)
    m_hi = Mk >> M_LO_BITS
    m_lo = Mk & ((1 << M_LO_BITS) - 1)
    pruned = take(W_bits.astype(np.uint16), pruned_cols)
    return Sk, Ek, m_hi, m_lo, pruned


def exponent_codebook(E_kept: np.ndarray):
    """(codebook: exponents by rank, rank_of: int [256], -1 where absent)."""
    counts = np.bincount(np.asarray(E_kept).ravel().astype(np.int64), minlength=256)
    present = [e for e in range(256) if counts[e] > 0]
    present.sort(key=lambda e: (-counts[e], e))
    rank_of = np.full(256, -1, dtype=np.int64)
    for r, e in enumerate(present):
        rank_of[e] = r
    return np.array(present, dtype=np.uint8), rank_of, counts


def unary_bits(ranks: np.ndarray) -> np.ndarray:
    """Concatenated codewords: rank r -> r zeros then a one. Returns a uint8 0/1 array."""
    ranks = np.asarray(ranks, dtype=np.int64)
    ends = np.cumsum(ranks + 1) - 1
    bits = np.zeros(int(ends[-1]) + 1 if len(ends) else 0, dtype=np.uint8)
    bits[ends] = 1
    return bits


def unary_decode(bits: np.ndarray, count: int) -> np.ndarray:
    """Ranks of the first `count` codewords: zeros counted up to each one."""
    ones = np.flatnonzero(np.asarray(bits))[:count]
    if len(ones) < count:
        raise ValueError("unary stream ends early")
    prev = np.concatenate(([-1], ones[:-1]))
    return ones - prev - 1


def bits_to_words(bits: np.ndarray) -> np.ndarray:
    """LSB-first packing of a 0/1 array into uint32 words (zero padded)."""
    n = len(bits)
    nw = (n + 31) // 32
    padded = np.zeros(nw * 32, dtype=np.uint32)
    padded[:n] = bits
    return (padded.reshape(nw, 32) << np.arange(32, dtype=np.uint32)).sum(axis=1, dtype=np.uint64).astype(np.uint32)


def words_to_bits(words: np.ndarray) -> np.ndarray:
    w = np.asarray(words, dtype=np.uint32)
    return ((w[:, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(np.uint8).ravel()


def nibbles_to_words(nib: np.ndarray) -> np.ndarray:
    """[N][L] nibbles -> [N][L/8] uint32, nibble i at bits 4*(i % 8)."""
    N, L = nib.shape
    n = nib.astype(np.uint32).reshape(N, L // 8, 8)
    w = np.zeros((N, L // 8), dtype=np.uint32)
    for i in range(8):
        w |= n[:, :, i] << np.uint32(4 * i)
    return w


def words_to_nibbles(w: np.ndarray) -> np.ndarray:
    N, L8 = w.shape
    out = np.empty((N, L8, 8), dtype=np.uint32)
    for i in range(8):
        out[:, :, i] = (w >> np.uint32(4 * i)) & 0xF
    return out.reshape(N, L8 * 8)


def pack(W_bits: np.ndarray, X_bits: np.ndarray):
    """Offline transform. Returns (buffer bytes, meta dict with offsets/sizes/codebook)."""
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    N, K = W_bits.shape
    assert K % 32 == 0
    c = column_norms(X_bits)
    keep = wanda_keep(W_bits, c)
    Sk, Ek, m_hi, m_lo, pruned = split_values(W_bits, keep)
    codebook, rank_of, counts = exponent_codebook(Ek)

    bitmap = np.zeros((N, K // 32), dtype=np.uint32)
    kb = keep.reshape(N, K // 32, 32).astype(np.uint32)
    for b in range(32):
        bitmap |= kb[:, :, b] << np.uint32(b)
    signmant = nibbles_to_words((Sk << M_HI_BITS) | m_hi)
    mlo = nibbles_to_words(m_lo)

    rows = []
    rowstart = np.zeros(N + 1, dtype=np.uint32)
    for n in range(N):
        words = bits_to_words(unary_bits(rank_of[Ek[n].astype(np.int64)]))
        pad = (-len(words)) % 4                      # 16-byte row alignment
        words = np.concatenate((words, np.zeros(pad, dtype=np.uint32)))
        rows.append(words)
        rowstart[n + 1] = rowstart[n] + len(words)
    stream = np.concatenate(rows) if rows else np.zeros(0, dtype=np.uint32)
    cb = np.zeros(256, dtype=np.uint8)
    cb[: len(codebook)] = codebook

    parts = [bitmap, signmant, stream, rowstart, cb, pruned.astype(np.uint16), mlo]
    raw = [np.ascontiguousarray(p).astype(p.dtype.newbyteorder("<")).tobytes() for p in parts]
    offs, total = layout.sections([len(r) for r in raw])
    buf = bytearray(total)
    for o, r in zip(offs, raw):
        buf[o:o + len(r)] = r
    meta = dict(N=N, K=K, offsets=offs, sizes=[len(r) for r in raw], total=total,
                n_symbols=len(codebook), codebook=codebook, keep=keep,
                stream_words=int(rowstart[-1]), counts=counts)
    return bytes(buf), meta


def _sections(buf: bytes, meta):
    N, K = meta["N"], meta["K"]
    o, s = meta["offsets"], meta["sizes"]
    get = lambda i, dt: np.frombuffer(buf, dtype=dt, count=s[i] // np.dtype(dt).itemsize, offset=o[i])
    bitmap = get(0, "<u4").reshape(N, K // 32)
    signmant = get(1, "<u4").reshape(N, K // 16)
    stream = get(2, "<u4")
    rowstart = get(3, "<u4")
    codebook = get(4, "u1")
    pruned = get(5, "<u2").reshape(N, K // 2)
    mlo = get(6, "<u4").reshape(N, K // 16)
    return bitmap, signmant, stream, rowstart, codebook, pruned, mlo


def _decode_common(buf: bytes, meta):
    N, K = meta["N"], meta["K"]
    bitmap, signmant, stream, rowstart, codebook, pruned, mlo = _sections(buf, meta)
    keep = ((bitmap[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool).reshape(N, K)
    if np.any(keep.sum(axis=1) != K // 2):
        raise ValueError("bitmap does not keep exactly K/2 values per row")
    sm = words_to_nibbles(signmant)
    S = sm >> M_HI_BITS
    m_hi = sm & ((1 << M_HI_BITS) - 1)
    E = np.empty((N, K // 2), dtype=np.uint32)
    nsym = meta["n_symbols"]
    for n in range(N):
        bits = words_to_bits(stream[rowstart[n]:rowstart[n + 1]])
        ranks = unary_decode(bits, K // 2)
        if np.any(ranks >= nsym):
            raise ValueError("unary rank beyond the codebook")
        E[n] = codebook[ranks]
    return keep, S, E, m_hi, pruned, words_to_nibbles(mlo)


def _scatter(keep, kept_vals, pruned_vals):
    N, K = keep.shape
    out = np.zeros((N, K), dtype=np.uint16)
    out[keep] = kept_vals.ravel()
    out[~keep] = pruned_vals.ravel()
    return out


def draft(buf: bytes, meta) -> np.ndarray:
    """Draft bf16 bits [N][K]: S, E, m_hi with zero low mantissa; pruned -> +0."""
    keep, S, E, m_hi, pruned, m_lo = _decode_common(buf, meta)
    kept = ((S << 15) | (E << 7) | (m_hi << M_LO_BITS)).astype(np.uint16)
    return _scatter(keep, kept, np.zeros_like(pruned))


def reconstruct(buf: bytes, meta) -> np.ndarray:
    """Target bf16 bits [N][K]: every original bit from speculation + verification data."""
    keep, S, E, m_hi, pruned, m_lo = _decode_common(buf, meta)
    kept = ((S << 15) | (E << 7) | (m_hi << M_LO_BITS) | m_lo).astype(np.uint16)
    return _scatter(keep, kept, pruned)


def speculation_bytes(meta) -> int:
    """Bytes the draft path must read: bitmap, sign+high mantissa, exponent stream, row starts, codebook."""
    return sum(meta["sizes"][:5])


def verification_bytes(meta) -> int:
    return sum(meta["sizes"][5:])


def exponent_stats(E_kept: np.ndarray):
    """(Shannon entropy in bits, mean unary code length in bits) of the kept exponents.

    "Cassandra" 3.3 quotes 2.58-2.64 bit entropy and a 2.85 bit mean for trained
    models. Pinned by closed forms (uniform, {2, 1, 1}, single symbol, a dyadic
    distribution) and the source-coding bound mean >= entropy.
    """
    _, rank_of, counts = exponent_codebook(E_kept)
    p = counts[counts > 0] / counts.sum()
    H = float(-(p * np.log2(p)).sum())
    ranks = rank_of[np.asarray(E_kept).ravel().astype(np.int64)]
    return H, float((ranks + 1).mean())


def dense_bytes(N: int, K: int) -> int:
    """Bytes of the uncompressed bf16 matrix (the draft/target streams are compared to it)."""
    return N * K * 2
