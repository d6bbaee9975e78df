"""Pins of the Cassandra-2 (MX shared-exponent) oracle against hand-derived values,
the exactness and truncation bound the method implies, and Cassandra-1's draft."""
import numpy as np

from oracle import cassandra, cassandra_mx
from oracle.numerics import bf16_bits_to_f64, bf16_fields
from quantized_gemv_unpack_gb300 import synth


def _fields(E, M, S=None):
    E = np.asarray(E, dtype=np.int64)[None, :]
    M = np.asarray(M, dtype=np.int64)[None, :]
    S = np.zeros_like(E) if S is None else np.asarray(S, dtype=np.int64)[None, :]
    return S, E, M


def test_hand_group():
    """One group of 32: exponents 121 x 30, 120, 119. The shared exponent is 121;
    1.1010101b * 2^(119-127) (sig 213) shifted right by 2 keeps 53 = 110101b, i.e.
    53 * 2^(121-134) = 0.0064697265625 against the original 0.006500244140625."""
    E = [121] * 30 + [120, 119]
    M = [0b0000000] * 30 + [0b1111111, 0b1010101]
    g, A = cassandra_mx.encode_groups(*_fields(E, M))
    assert g.tolist() == [[121]]
    assert A[0, :30].tolist() == [128] * 30
    assert A[0, 30] == 255 >> 1 == 127                     # 1.1111111b, one bit dropped
    assert A[0, 31] == 213 >> 2 == 53
    assert np.ldexp(53.0, 121 - 134) == 0.0064697265625
    assert np.ldexp(213.0, 119 - 127 - 7) == 0.006500244140625
    # draft magnitude = top 4 bits: 8 for the aligned ones, 7 and 3 for the shifted ones
    assert (A[0] >> 4).tolist() == [8] * 30 + [7, 3]


def test_far_below_the_shared_exponent_reads_zero():
    g, A = cassandra_mx.encode_groups(*_fields([130] + [121] * 31, [0] * 32))
    assert g[0, 0] == 130 and A[0, 0] == 128 and np.all(A[0, 1:] == 0)   # shift 9 >= 8


def test_subnormal_group_is_exact():
    """E = 0 values (sig = M at exponent 1) in a group of subnormals keep every bit."""
    M = np.arange(32) * 3 % 128
    g, A = cassandra_mx.encode_groups(*_fields([0] * 32, M))
    assert g[0, 0] == 1 and np.array_equal(A[0], M)
    assert np.array_equal(np.ldexp(A[0].astype(float), 1 - 134), bf16_bits_to_f64(M.astype(np.uint16)))


def _pack(N=24, K=256, seed=11):
    g = synth.rng(seed)
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, 16, K)
    buf, meta = cassandra_mx.pack(W, X)
    return W, X, buf, meta


def test_target_is_exact_at_the_shared_exponent_and_within_one_unit_below():
    W, X, buf, meta = _pack()
    N, K = W.shape
    keep = meta["keep"]
    tgt = cassandra_mx.reconstruct(buf, meta)
    # pruned values come back bit for bit
    assert np.array_equal(tgt[~keep], W[~keep])
    # kept values: exact where the exponent is the group's maximum, below by less than 2^(g - 134) elsewhere
    S, E, M = bf16_fields(W)
    Ek = E[keep].reshape(N, K // 2).astype(np.int64)
    e = np.maximum(Ek, 1)
    gmax = np.repeat(e.reshape(N, K // 64, 32).max(axis=2), 32, axis=1)
    orig = bf16_bits_to_f64(W[keep].reshape(N, K // 2))
    got = bf16_bits_to_f64(tgt[keep].reshape(N, K // 2))
    at = e == gmax
    assert at.any() and (~at).any()
    assert np.array_equal(got[at], orig[at])
    gap = np.abs(orig) - np.abs(got)
    assert np.all(gap >= 0) and np.all(gap < np.ldexp(1.0, gmax - 134))
    assert np.all(np.signbit(got) == np.signbit(orig))


def test_draft_matches_cassandra1_where_exponent_is_the_shared_one():
    W, X, buf, meta = _pack(seed=12)
    N, K = W.shape
    keep = meta["keep"]
    buf1, meta1 = cassandra.pack(W, X)
    assert np.array_equal(meta1["keep"], keep)              # same Wanda selection
    d1 = cassandra.draft(buf1, meta1)
    d2 = cassandra_mx.draft(buf, meta)
    assert np.all(d2[~keep] == 0)
    _, E, _ = bf16_fields(W)
    Ek = np.maximum(E[keep].reshape(N, K // 2).astype(np.int64), 1)
    at = (Ek == np.repeat(Ek.reshape(N, K // 64, 32).max(axis=2), 32, axis=1)) & (E[keep].reshape(N, K // 2) > 0)
    assert np.array_equal(d2[keep].reshape(N, K // 2)[at], d1[keep].reshape(N, K // 2)[at])


def test_negative_zero_keeps_its_sign():
    """A row of -0.0: every score is 0, so the lower half of the columns is kept (ties keep
    the lower column). Kept -0 decodes to -0 in both paths; pruned -0 is +0 in the draft
    and its raw bits in the target."""
    W = np.full((1, 64), 0x8000, np.uint16)
    X = np.full((4, 64), 0x3F80, np.uint16)
    buf, meta = cassandra_mx.pack(W, X)
    assert meta["keep"][0, :32].all() and not meta["keep"][0, 32:].any()
    assert np.all(cassandra_mx.reconstruct(buf, meta) == 0x8000)
    d = cassandra_mx.draft(buf, meta)
    assert np.all(d[0, :32] == 0x8000) and np.all(d[0, 32:] == 0)


def test_bit_accounting():
    """Speculation data 1 (bitmap) + 1/2 (signs) + 2 (4-bit magnitudes) + 1/8 (shared exponents)
    = 3.625 bits per weight; with the verification data (4-bit low magnitudes of the kept half,
    raw bf16 of the pruned half) 13.625 of bf16's 16."""
    N, K = 16, 1024
    sizes = cassandra_mx.section_sizes(N, K)
    assert sum(sizes[:4]) * 8 / (N * K) == 3.625
    assert sum(sizes) * 8 / (N * K) == 13.625
