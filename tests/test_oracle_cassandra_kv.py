"""Pins of the online KV encoder oracle: magnitude pruning against a brute-force sort, the
fixed-codebook unary stream against a hand-built one, the lossless round trip through the
Cassandra-1 decoders, and the slot overflow rule."""
import numpy as np

from oracle import cassandra, cassandra_kv as kv
from oracle.numerics import bf16_bits_to_f64, bf16_fields
from quantized_gemv_unpack_gb300 import synth


def test_magnitude_keep_is_a_sort():
    g = synth.rng(31)
    W = synth.to_bf16_bits(g.standard_normal((12, 64)).astype(np.float32))
    W[0, :8] = W[0, 8]                                  # ties in row 0
    W[1, 3] = 0x7FC0                                    # NaN: kept as if +inf
    W[1, 9] = 0xFF80                                    # -inf
    W[2, :] = 0x8000                                    # all -0: the lower half is kept
    keep = kv.magnitude_keep(W)
    for n in range(12):
        mag = np.abs(bf16_bits_to_f64(W[n]))
        mag = np.where(np.isnan(mag), np.inf, mag)
        order = sorted(range(64), key=lambda j: (-mag[j], j))
        assert set(np.flatnonzero(keep[n])) == set(order[:32]), n
    assert keep[1, 3] and keep[1, 9] and keep[2, :32].all() and not keep[2, 32:].any()


def test_codebook_from_hand_case():
    cb = kv.codebook_from(np.array([121, 120, 121, 119, 121, 120]))
    assert cb[:3].tolist() == [121, 120, 119]
    assert cb[3:].tolist() == [e for e in range(256) if e not in (119, 120, 121)]


def test_fixed_codebook_stream_by_hand():
    """One row of 64 values, kept in order with exponents 121, 120, 119, 121, ... (the other 28
    kept values at 121); codebook 121, 120, 119, ...: codes 1, 01, 001, 1, 1 ... -> bits
    1 01 001 1 ... = word 0b...1_1_100_10_1 read LSB first."""
    E = np.full(32, 121)
    E[1], E[2] = 120, 119
    W = np.zeros((1, 64), np.uint16)
    W[0, :32] = ((E << 7) | 0x55).astype(np.uint16)     # large values: kept
    W[0, 32:] = 0x0001                                  # tiny subnormals: pruned
    cb = np.array([121, 120, 119] + [e for e in range(256) if e not in (119, 120, 121)], np.uint8)
    buf, meta, fits = kv.pack(W, cb, 4)
    assert fits.all() and meta["keep"][0, :32].all()
    o = meta["offsets"]
    stream = np.frombuffer(buf, "<u4", 4, o[2])
    bits = "1" + "01" + "001" + "1" * 29                # LSB first, 35 bits
    assert stream[0] == int(bits[:32][::-1], 2) and stream[1] == int(bits[32:][::-1], 2) and stream[2] == 0
    assert np.frombuffer(buf, "<u4", 2, o[3]).tolist() == [0, 4]
    assert np.array_equal(np.frombuffer(buf, "u1", 256, o[4]), cb)


def test_round_trip_through_the_cassandra_decoders():
    g = synth.rng(32)
    W = synth.to_bf16_bits((g.standard_normal((40, 256)) * 0.3).astype(np.float32))
    W[5, 17] = 0x7F80                                   # +inf among ordinary values
    cb = kv.codebook_from(bf16_fields(W[:4])[1])        # "calibration" on the first tokens
    buf, meta, fits = kv.pack(W, cb, 48)
    assert fits.all()
    assert np.array_equal(cassandra.reconstruct(buf, meta), W)
    d = cassandra.draft(buf, meta)
    keep = meta["keep"]
    assert np.array_equal(d[keep], W[keep] & 0xFFF0) and np.all(d[~keep] == 0)


def test_slot_overflow_is_reported():
    W = np.zeros((2, 64), np.uint16)
    W[0, :] = 0x3F80                                    # exponent 127
    W[1, :] = 0x3C00                                    # exponent 120
    cb = kv.codebook_from(np.array([127]))              # 120 gets rank 121: a 122-bit code per value
    _, _, fits = kv.pack(W, cb, 4)
    assert fits.tolist() == [True, False]
