"""Bit-level number conversions used by the oracle (float64 <-> fp16, bf16 fields).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The fp16 conversion is written out from the IEEE-754 binary16 definition
(1 sign bit, 5 exponent bits with bias 15, 10 fraction bits, subnormals below
2**-14, overflow to infinity), rounding the exact float64 value to nearest,
ties to even, in one step (no intermediate float32 rounding).
"""
from __future__ import annotations

import numpy as np

_F64_FRAC = np.uint64((1 << 52) - 1)


def f64_to_f16_bits(a) -> np.ndarray:
    """Round float64 values to binary16 (nearest, ties to even); return uint16 bits."""
    a = np.asarray(a, dtype=np.float64)
    bits = a.view(np.uint64).astype(np.uint64)
    sign = ((bits >> np.uint64(63)) & np.uint64(1)).astype(np.uint64)
    exp = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    frac = bits & _F64_FRAC
    # significand with the implicit bit (53 bits) for normal float64 inputs
    sig = np.where(exp > 0, frac | np.uint64(1 << 52), frac).astype(np.uint64)
    e_unb = np.where(exp > 0, exp - 1023, -1022)          # value = sig * 2**(e_unb - 52)

    out = np.zeros(a.shape, dtype=np.uint64)

    # right shift that brings the significand to units of the binary16 ulp:
    # normal binary16 (e_unb >= -14): ulp = 2**(e_unb - 10)  -> shift 42
    # subnormal binary16: ulp = 2**-24 -> shift = (-24) - (e_unb - 52)
    shift = np.where(e_unb >= -14, 42, 28 - e_unb).astype(np.int64)
    big = shift >= 64
    sh = np.clip(shift, 0, 63).astype(np.uint64)
    kept = np.where(big, np.uint64(0), sig >> sh)
    rem = np.where(big, sig, sig - (kept << sh))
    half = np.where(big, np.uint64(0), np.uint64(1) << (sh - np.uint64(1)))
    # for shift >= 64 the value is below 2**-25 < half an ulp -> rounds to 0
    round_up = (~big) & ((rem > half) | ((rem == half) & ((kept & np.uint64(1)) == 1)))
    q = kept + round_up.astype(np.uint64)

    normal = e_unb >= -14
    # normal: q in [1024, 2048]; encode exponent field e_unb + 15, carry allowed
    e_field = (e_unb + 15).astype(np.int64)
    enc_normal = (np.clip(e_field - 1, 0, None).astype(np.uint64) << np.uint64(10)) + q
    enc_sub = q  # subnormal count (a carry into 1024 yields the smallest normal)
    enc = np.where(normal, enc_normal, enc_sub)
    overflow = (enc >= np.uint64(0x7C00)) | (exp == 0x7FF)
    enc = np.where(overflow, np.uint64(0x7C00), enc)
    isnan = (exp == 0x7FF) & (frac != 0)
    enc = np.where(isnan, np.uint64(0x7E00), enc)
    out = enc | (sign << np.uint64(15))
    return out.astype(np.uint16)


def f16_bits_to_f64(b) -> np.ndarray:
    """Exact value of binary16 bit patterns as float64."""
    b = np.asarray(b, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    mag = np.where(e == 0, f * 2.0 ** -24,
                   np.where(e == 31, np.where(f == 0, np.inf, np.nan),
                            (1024.0 + f) * np.exp2((e - 25).astype(np.float64))))
    return sign * mag


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact value of bfloat16 bit patterns as float64 (via the float32 with the same top bits)."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_fields(b):
    """Split bfloat16 bits into (S, E, M): [1 sign][8 exponent][7 mantissa] ("Cassandra", 3.1)."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32)
    return (b >> 15) & 1, (b >> 7) & 0xFF, b & 0x7F


def bf16_from_fields(S, E, M) -> np.ndarray:
    S = np.asarray(S, dtype=np.uint32)
    E = np.asarray(E, dtype=np.uint32)
    M = np.asarray(M, dtype=np.uint32)
    return ((S << 15) | (E << 7) | M).astype(np.uint16)


def bf16_value_from_fields(S, E, M) -> np.ndarray:
    """(-1)**S * 2**(E-127) * (1 + M/128) for normal E; the bf16 layout of "Cassandra" 3.1.

    Exponent field 0 (zero/subnormal) uses 2**-126 * (M/128), field 255 gives inf/nan,
    as IEEE binary formats define them.
    """
    S = np.asarray(S, dtype=np.int64)
    E = np.asarray(E, dtype=np.int64)
    M = np.asarray(M, dtype=np.float64)
    sgn = np.where(S == 1, -1.0, 1.0)
    normal = (1.0 + M / 128.0) * np.exp2((E - 127).astype(np.float64))
    sub = (M / 128.0) * 2.0 ** -126
    special = np.where(M == 0, np.inf, np.nan)
    return sgn * np.where(E == 0, sub, np.where(E == 255, special, normal))
