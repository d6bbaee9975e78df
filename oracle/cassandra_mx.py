"""Cassandra-2: the MX shared-exponent split. TEST INFRASTRUCTURE ONLY.

Written from "Cassandra: ... self-speculative decoding" (cnblogs summary),
section 3.3, the third encoding it compares: instead of coding each exponent,
a group of neighbouring values (about 32) shares one maximum exponent and every
value's mantissa is shifted right by the difference between its own exponent
and the shared one; this compresses more and decodes faster, and the shift
drops low bits of the smaller values (slightly lossy).

Value pruning and the bitmap are those of Cassandra-1 (``oracle.cassandra``,
section 3.2 step 1): the Wanda-selected half of every row is kept, pruned values
go to the verification data as raw bf16 bits.

Readings (the page gives only the idea):
* a group is 32 consecutive kept values of a row, in column order (K/2 must be
  a multiple of 32, so K a multiple of 64);
* a kept value with fields (S, E, M) has the 8-bit significand
  sig = 128 + M for E > 0 and sig = M for E = 0 (subnormal), at exponent
  e = max(E, 1); the group's shared exponent is g = max e over the group;
* the aligned magnitude is A = sig >> (g - e), truncated (0 once the shift
  reaches 8), so the value A * 2^(g - 134) equals the original when e = g and
  is below it by less than 2^(g - 134) otherwise;
* the speculation data holds the sign and the high 4 bits D = A >> 4; the
  verification data holds the low 4 bits L = A & 15. Draft value
  (-1)^S * D * 2^(g - 130), target value (-1)^S * A * 2^(g - 134); both are
  exactly representable in bf16. When e = g the draft equals Cassandra-1's
  (sign, exponent and the high 3 mantissa bits, low bits zero);
* exponent 255 (Inf/NaN) is an ordinary exponent here: MX has no special
  values, and bf16 weights of a model carry none; in a group whose shared
  exponent is 255 a value with A >= 128 is at least 2^128, beyond bf16's range,
  and decodes to +-Inf (the decode arithmetic overflows).

Layout (sections 256-byte aligned, ``oracle.layout.sections``):
  0 bitmap : N x K/32 uint32, bit (j % 32) of word j // 32 = kept(n, j)
  1 gexp   : N x K/64 uint8, shared exponent g of each group of the row
  2 signs  : N x K/64 uint32, bit (i % 32) of word i // 32 = S of kept value i
  3 dnib   : N x K/16 uint32, nibble i (bits 4(i % 8)..) = D of kept value i
  4 lnib   : N x K/16 uint32, nibble i = L of kept value i
  5 pruned : N x K/2 uint16, raw bf16 bits of the pruned values, column order
Sections 0-3 are the speculation data, 4-5 the verification data.
"""
from __future__ import annotations

import numpy as np

from . import layout
from .cassandra import column_norms, nibbles_to_words, wanda_keep, words_to_nibbles
from .numerics import bf16_fields

GROUP = 32


def section_sizes(N: int, K: int):
    return [N * K // 32 * 4, N * K // 64, N * K // 64 * 4, N * K // 16 * 4, N * K // 16 * 4, N * K // 2 * 2]


def encode_groups(S, E, M):
    """Kept-order fields [N][K/2] -> (g [N][K/64], A [N][K/2]) by the group rule above."""
    N, H = E.shape
    e = np.maximum(E.astype(np.int64), 1)
    sig = np.where(E > 0, 128, 0).astype(np.int64) + M.astype(np.int64)
    g = e.reshape(N, H // GROUP, GROUP).max(axis=2)
    shift = np.repeat(g, GROUP, axis=1) - e
    A = np.where(shift < 8, sig >> np.minimum(shift, 63), 0)
    return g, A


def pack(W_bits: np.ndarray, X_bits: np.ndarray):
    """Offline transform. Returns (buffer bytes, meta dict)."""
    W_bits = np.asarray(W_bits, dtype=np.uint16)
    N, K = W_bits.shape
    assert K % 64 == 0
    keep = wanda_keep(W_bits, column_norms(X_bits))
    S, E, M = bf16_fields(W_bits)
    kept_cols = np.nonzero(keep)[1].reshape(N, K // 2)
    pruned_cols = np.nonzero(~keep)[1].reshape(N, K // 2)
    take = lambda a, cols: np.take_along_axis(a, cols, axis=1)
    Sk, Ek, Mk = take(S, kept_cols), take(E, kept_cols), take(M, kept_cols)
    g, A = encode_groups(Sk, Ek, Mk)

    bitmap = np.zeros((N, K // 32), dtype=np.uint32)
    kb = keep.reshape(N, K // 32, 32).astype(np.uint32)
    for b in range(32):
        bitmap |= kb[:, :, b] << np.uint32(b)
    signs = np.zeros((N, K // 64), dtype=np.uint32)
    sb = Sk.reshape(N, K // 64, 32).astype(np.uint32)
    for b in range(32):
        signs |= sb[:, :, b] << np.uint32(b)
    parts = [bitmap, g.astype(np.uint8), signs, nibbles_to_words(A >> 4), nibbles_to_words(A & 15),
             take(W_bits, pruned_cols).astype(np.uint16)]
    raw = [np.ascontiguousarray(p).astype(p.dtype.newbyteorder("<")).tobytes() for p in parts]
    assert [len(r) for r in raw] == section_sizes(N, K)
    offs, total = layout.sections([len(r) for r in raw])
    buf = bytearray(total)
    for o, r in zip(offs, raw):
        buf[o:o + len(r)] = r
    meta = dict(N=N, K=K, offsets=offs, sizes=[len(r) for r in raw], total=total, keep=keep)
    return bytes(buf), meta


def _read(buf: bytes, meta):
    N, K = meta["N"], meta["K"]
    o = meta["offsets"]
    bitmap = np.frombuffer(buf, "<u4", N * K // 32, o[0]).reshape(N, K // 32)
    g = np.frombuffer(buf, "u1", N * K // 64, o[1]).reshape(N, K // 64).astype(np.int64)
    signs = np.frombuffer(buf, "<u4", N * K // 64, o[2]).reshape(N, K // 64)
    D = words_to_nibbles(np.frombuffer(buf, "<u4", N * K // 16, o[3]).reshape(N, K // 16)).astype(np.int64)
    L = words_to_nibbles(np.frombuffer(buf, "<u4", N * K // 16, o[4]).reshape(N, K // 16)).astype(np.int64)
    pruned = np.frombuffer(buf, "<u2", N * K // 2, o[5]).reshape(N, K // 2)
    keep = ((bitmap[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool).reshape(N, K)
    S = ((signs[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(N, K // 2).astype(np.int64)
    return keep, g, S, D, L, pruned


def _bf16_bits_of(values: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float64 values that bf16 represents exactly (checked), values
    of magnitude 2^128 or more as +-Inf."""
    values = np.asarray(values, dtype=np.float64)
    with np.errstate(over="ignore"):
        f = values.astype(np.float32)
    fin = np.isfinite(f)
    assert np.array_equal(f[fin].astype(np.float64), values[fin]), "value not representable"
    assert np.all(np.abs(values[~fin]) >= 2.0 ** 128), "overflow below bf16's range"
    bits = f.view(np.uint32)
    assert not np.any(bits & 0xFFFF), "value not representable in bf16"
    return (bits >> 16).astype(np.uint16)


def _scatter(keep, kept_bits, pruned_bits):
    N, K = keep.shape
    out = np.zeros((N, K), dtype=np.uint16)
    out[keep] = kept_bits.ravel()
    out[~keep] = pruned_bits.ravel()
    return out


def kept_values(buf: bytes, meta, target: bool) -> np.ndarray:
    """float64 [N][K/2]: the decoded kept values (draft: sign and D; target: sign and A)."""
    keep, g, S, D, L, _ = _read(buf, meta)
    ge = np.repeat(g, GROUP, axis=1)
    mag = np.ldexp(((D << 4) | L).astype(np.float64), ge - 134) if target else np.ldexp(D.astype(np.float64), ge - 130)
    return np.where(S == 1, -mag, mag)


def draft(buf: bytes, meta) -> np.ndarray:
    """bf16 bits [N][K] of the draft weights: decoded kept values, pruned positions +0."""
    keep = _read(buf, meta)[0]
    return _scatter(keep, _bf16_bits_of(kept_values(buf, meta, False)), np.zeros(int((~keep).sum()), np.uint16))


def reconstruct(buf: bytes, meta) -> np.ndarray:
    """bf16 bits [N][K] of the target weights: decoded kept values, raw pruned values."""
    keep, _, _, _, _, pruned = _read(buf, meta)
    return _scatter(keep, _bf16_bits_of(kept_values(buf, meta, True)), pruned)


def speculation_bytes(meta) -> int:
    return sum(meta["sizes"][:4])


def verification_bytes(meta) -> int:
    return sum(meta["sizes"][4:])
