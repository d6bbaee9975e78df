"""Pins for the oracle's number conversions, ternary and INT4 quantizers and packed layouts.

Each check is fixed by something other than the oracle itself: a closed form
derived by hand from the pages' formulas, a library routine (NumPy's float16
conversion), exact rational arithmetic, or the pages' own bit accounting.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import int4, layout, numerics, ternary
from oracle.matvec import matvec
from quantized_gemv_unpack_gb300 import synth

from conftest import GOLDEN

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------- fp16

def test_fp16_rounding_matches_numpy():
    g = np.random.default_rng(7)
    a = g.standard_normal(400_000) * 10.0 ** g.uniform(-9, 5, 400_000)
    ours = numerics.f64_to_f16_bits(a)
    ref = a.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("t", [0.5, 0.5 + 2.0 ** -30, 0.5 - 2.0 ** -30])
def test_fp16_rounding_halfway(t):
    """Exact float64 halfway points (and a hair either side): a float32 detour would get these wrong."""
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    v = numerics.f16_bits_to_f64(h)
    a = v + (numerics.f16_bits_to_f64(h + 1) - v) * t
    assert np.array_equal(numerics.f64_to_f16_bits(a), a.astype(np.float16).view(np.uint16))


def test_fp16_decode_all_patterns():
    b = np.arange(0x7C00, dtype=np.uint16)
    assert np.array_equal(numerics.f16_bits_to_f64(b), b.view(np.float16).astype(np.float64))


# ----------------------------------------------------------------------------- bf16 layout

def test_bf16_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "bf16_worked_example.json")))
    bits = int(ex["bits"].replace(" ", ""), 2)
    S, E, M = numerics.bf16_fields(np.array([bits], dtype=np.uint16))
    assert (int(S[0]), int(E[0])) == (ex["S"], ex["E"])
    assert int(M[0]) == int(ex["mantissa_bits"], 2)
    assert int(M[0]) / 128 == ex["mantissa_fraction"]
    assert numerics.bf16_bits_to_f64(np.array([bits], np.uint16))[0] == ex["value"]
    assert numerics.bf16_value_from_fields(S, E, M)[0] == ex["value"]
    # bf16 is the top half of float32: the library's own float32 agrees
    assert np.array([ex["value"]], np.float32).view(np.uint32)[0] >> 16 == bits
    hi = int(ex["truncated_high_bits"], 2)
    assert int(M[0]) >> 4 == hi
    trunc = numerics.bf16_from_fields(S, E, np.array([hi << 4]))
    assert numerics.bf16_bits_to_f64(trunc)[0] == ex["truncated_value"]


# ----------------------------------------------------------------------------- ternary

def _one_block(vals):
    w = np.zeros((1, 128), np.float32)
    w[0, : len(vals)] = vals
    return w


def test_ternary_threshold_and_sign():
    # 64 values of +-1 and 64 of +-v: mean|w| = 0.5 + 0.5 v (+1e-8).
    # v = 0.3: v / mean = 0.4615 -> 0 ; v = 0.4: 0.5714 -> +-1.  Negative inputs give -1.
    for v, expect in [(0.3, 0), (0.4, 1)]:
        w = np.array([1.0, -1.0] * 32 + [v, -v] * 32, np.float32)[None, :]
        q, s_star, s16 = ternary.quantize(w)
        assert list(q[0, :64]) == [1, -1] * 32
        assert list(q[0, 64:]) == [expect, -expect] * 32
        mean = (64 + 64 * float(np.float32(v))) / 128
        assert s_star[0, 0] == pytest.approx(mean + 1e-8, rel=0, abs=1e-15)
        assert s16[0, 0] == numerics.f64_to_f16_bits(np.array([mean + 1e-8]))[0]


def test_ternary_single_outlier_and_constant_block():
    # one nonzero value a: mean = a/128, a/mean = 128 -> clamps to sign(a)
    q, s, _ = ternary.quantize(_one_block([-0.37]))
    assert q[0, 0] == -1 and not q[0, 1:].any()
    assert s[0, 0] == pytest.approx(0.37 / 128 + 1e-8, rel=1e-7)
    # a constant block c: w/scale = c/(c + 1e-8) -> 1
    q, _, _ = ternary.quantize(np.full((1, 128), 0.02, np.float32))
    assert (q == 1).all()


def test_ternary_all_zero_block_has_no_nan():
    w = np.zeros((2, 256), np.float32)
    w[1, 128:] = 0.5
    q, s_star, s16 = ternary.quantize(w)
    assert not q[0].any() and not q[1, :128].any()
    assert s_star[0, 0] == 1e-8 and s16[0, 0] == 0          # 1e-8 is below half the smallest fp16 subnormal
    assert np.isfinite(ternary.dequant(q, s16)).all()


def _round_half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def test_ternary_exact_rational_brute_force():
    """8 x 128: exact-rational block_ternary against the float64 oracle."""
    w = synth.student_t4(synth.rng(11), (8, 128))
    q, s_star, s16 = ternary.quantize(w)
    for n in range(8):
        vals = [Fraction(float(v)) for v in w[n]]
        scale = sum(abs(v) for v in vals) / 128 + Fraction(1e-8)
        for k in range(128):
            r = vals[k] / scale
            assert abs(float(r) % 1.0 - 0.5) > 1e-9          # no near-ties in this draw
            assert q[n, k] == max(-1, min(1, _round_half_even(r)))
        assert s16[n, 0] == numerics.f64_to_f16_bits(np.array([float(scale)]))[0]


def test_ternary_pack_layout_hand_word():
    # k=0: +1 -> code 01 at bit 0; k=1: -1 -> code 10 at bit 16 (odd columns in the high half)
    # k=2: -1 -> code 10 at bit 2; k=15: +1 -> code 01 at bit 30
    q = np.zeros((1, 128), np.int8)
    q[0, [0, 1, 2, 15]] = [1, -1, -1, 1]
    buf = ternary.pack(q, np.zeros((1, 1), np.uint16))
    word = np.frombuffer(buf, "<u4", count=1)[0]
    assert word == (0b01 << 0) | (0b10 << 16) | (0b10 << 2) | (0b01 << 30)


def test_ternary_record_layout_hand_position():
    # N=20 rows (2 row groups, the second padded), K=1280 (10 blocks: steps of 8 and 2).
    # q = +1 at row 17, column 1100: group 1, row 1 of the group; block 8 -> step 1 (nbk = 2),
    # block 0 of the step; column 76 of the block -> word 4, bit 12 (even column).
    # byte offset = 1*16*(1280/4) + 16*8*32 + 1*2*32 + 0*32 + 4*4 = 5120 + 4096 + 64 + 16 = 9296
    q = np.zeros((20, 1280), np.int8)
    q[17, 1100] = 1
    buf = ternary.pack(q, np.zeros((20, 10), np.uint16))
    words = np.frombuffer(buf, "<u4", count=32 * 1280 // 16)
    assert np.flatnonzero(words).tolist() == [9296 // 4]
    assert words[9296 // 4] == 1 << 12
    # the padded rows 20..31 are all-zero codes
    assert len(buf) >= 32 * 1280 // 4


def test_ternary_pack_roundtrip_and_size():
    g = synth.rng(3)
    q = g.integers(-1, 2, (5, 384)).astype(np.int8)
    s16 = g.integers(0, 0x7BFF, (5, 3)).astype(np.uint16)
    buf = ternary.pack(q, s16)
    q2, s2 = ternary.unpack(buf, 5, 384)
    assert np.array_equal(q, q2) and np.array_equal(s16, s2)
    # bytes of codes + scales = 2 + 16/128 bits per weight (the pages' 2 + 16/256 accounting with block 128)
    bpw = json.load(open(os.path.join(GOLDEN, "bits_per_weight.json")))
    iq = bpw["iq2_xxs"]
    assert iq["data_bits"] + iq["scale_bits"] / iq["block"] == iq["bits_per_weight"]
    t = bpw["this_library"]["ternary_block128_fp16"]
    assert layout.payload_bytes(32, 384, 2) * 8 / (32 * 384) == t["bits_per_weight"]
    t = bpw["this_library"]["int4_group128_fp16"]
    assert layout.payload_bytes(32, 384, 4) * 8 / (32 * 384) == t["bits_per_weight"]
    # the stored sections add nothing to that payload when rows come in groups of 16 and K in steps of 1024
    assert sum(layout.ternary_sizes(32, 2048)) == layout.payload_bytes(32, 2048, 2)
    assert sum(layout.int4_sizes(48, 5120)) == layout.payload_bytes(48, 5120, 4)


def test_scale_records_hand_placed():
    """Section 1 stores scales in the order of the code records: (row 17, block 9) of a
    20 x 1280 matrix is row 1 of group 1, block 1 of step 1; with 2 steps per row that is
    element ((1 * 2 + 1) * 128) + 1 * 8 + 1 = 393."""
    assert layout.scale_index(17, 9, 1280) == 393
    s16 = np.zeros((20, 10), np.uint16)
    s16[17, 9] = 0x3C00
    flat = layout.scale_records_from_rows(s16, 1280)
    assert flat.size == 2 * 2 * 128 and np.flatnonzero(flat).tolist() == [393]
    assert np.array_equal(layout.rows_from_scale_records(flat, 20, 1280), s16)
    q = np.zeros((20, 1280), np.int8)
    buf = ternary.pack(q, s16)
    offs, _ = layout.sections(layout.ternary_sizes(20, 1280))
    assert buf[offs[1] + 2 * 393:offs[1] + 2 * 393 + 2] == bytes([0x00, 0x3C])


def test_ternary_unpack_rejects_code_11():
    q = np.zeros((1, 128), np.int8)
    buf = bytearray(ternary.pack(q, np.zeros((1, 1), np.uint16)))
    buf[0] = 0b11
    with pytest.raises(ValueError):
        ternary.unpack(bytes(buf), 1, 128)


# ----------------------------------------------------------------------------- INT4

def test_int4_group_max_reaches_seven():
    w = synth.student_t4(synth.rng(5), (16, 512))
    q, s_star, _ = int4.quantize(w)
    g = w.reshape(16, 4, 128)
    qg = q.reshape(16, 4, 128)
    am = np.abs(g).argmax(axis=2)
    top = np.take_along_axis(qg, am[:, :, None], axis=2)[:, :, 0]
    top_w = np.take_along_axis(g, am[:, :, None], axis=2)[:, :, 0]
    assert np.array_equal(top, np.where(top_w > 0, 7, -7))
    assert q.min() >= -7 and q.max() <= 7


def test_int4_hand_group():
    # max|w| = 0.7 -> scale = 0.1 (float64 0.7/7); 0.26/0.1 = 2.6 -> 3; -0.14/0.1 = -1.4 -> -1; 0.04 -> 0
    w = np.zeros((1, 128), np.float32)
    w[0, :4] = [0.7, 0.26, -0.14, 0.04]
    q, s_star, _ = int4.quantize(w)
    assert list(q[0, :4]) == [7, 3, -1, 0] and not q[0, 4:].any()
    assert s_star[0, 0] == float(np.float32(0.7)) / 7


def test_int4_all_zero_group():
    q, s_star, s16 = int4.quantize(np.zeros((1, 128), np.float32))
    assert not q.any() and s_star[0, 0] == 0 and s16[0, 0] == 0


def test_int4_exact_rational_brute_force():
    w = synth.student_t4(synth.rng(12), (8, 128))
    q, _, _ = int4.quantize(w)
    for n in range(8):
        vals = [Fraction(float(v)) for v in w[n]]
        scale = max(abs(v) for v in vals) / 7
        for k in range(128):
            r = vals[k] / scale
            assert abs(float(r) % 1.0 - 0.5) > 1e-9
            assert q[n, k] == max(-7, min(7, _round_half_even(r)))


def test_int4_pack_layout_hand_word():
    # k=0: -7 -> nibble 0x9 at bit 0; k=1: 7 -> 0x7 at bit 16; k=6: 1 -> bit 12; k=7: -1 -> 0xF at bit 28
    q = np.zeros((1, 128), np.int8)
    q[0, [0, 1, 6, 7]] = [-7, 7, 1, -1]
    buf = int4.pack(q, np.zeros((1, 1), np.uint16))
    word = np.frombuffer(buf, "<u4", count=1)[0]
    assert word == 0x9 | (0x7 << 16) | (0x1 << 12) | (0xF << 28)


def test_int4_pack_roundtrip():
    g = synth.rng(4)
    q = g.integers(-7, 8, (3, 256)).astype(np.int8)
    s16 = g.integers(0, 0x7BFF, (3, 2)).astype(np.uint16)
    q2, s2 = int4.unpack(int4.pack(q, s16), 3, 256)
    assert np.array_equal(q, q2) and np.array_equal(s16, s2)


# ----------------------------------------------------------------------------- matvec

def test_matvec_exact_rational_brute_force():
    g = synth.rng(21)
    w = synth.student_t4(g, (8, 128))
    q, _, s16 = ternary.quantize(w)
    wh = ternary.dequant(q, s16)
    x = numerics.bf16_bits_to_f64(synth.activations_bf16(g, (3, 128)))
    y, B = matvec(wh, x)
    for m in range(3):
        for n in range(8):
            exact = sum(Fraction(float(wh[n, k])) * Fraction(float(x[m, k])) for k in range(128))
            babs = sum(abs(Fraction(float(wh[n, k])) * Fraction(float(x[m, k]))) for k in range(128))
            assert abs(Fraction(float(y[m, n])) - exact) <= Fraction(1, 10 ** 12) * babs
            assert float(B[m, n]) == pytest.approx(float(babs), rel=1e-12)


def test_matvec_unit_vector_selects_a_column_and_ones_sum():
    g = synth.rng(22)
    w = synth.student_t4(g, (6, 256))
    q, _, s16 = ternary.quantize(w)
    wh = ternary.dequant(q, s16)
    x = np.zeros((1, 256))
    x[0, 131] = 1.0
    y, _ = matvec(wh, x)
    assert np.array_equal(y[0], wh[:, 131])               # not a transposed operand
    # a block of one positive constant quantizes to all +1: y = s * sum(x)
    wc = np.full((1, 128), 0.02, np.float32)
    qc, _, sc = ternary.quantize(wc)
    xr = g.standard_normal((1, 128))
    yc, _ = matvec(ternary.dequant(qc, sc), xr)
    assert yc[0, 0] == pytest.approx(numerics.f16_bits_to_f64(sc)[0, 0] * xr.sum(), rel=1e-14)
