"""Pins of the oracle's byte-lookup ternary layout (CPU only).

The pages fix the ternary codes (00 = 0, 01 = +1, 10 = -1, "Ternary Bonsai 2"
section 1.2) and one fp16 scale per block of 128, but no byte order; this
library's lookup layout is stated in its header and in ``oracle.layout``. The
hand-placed cases below were worked out by hand from that statement, so a
transposed index, a wrong rotation direction or a swapped half shows up as a
wrong byte.
"""
import numpy as np
import pytest

from oracle import layout, ternary
from quantized_gemv_unpack_gb300 import synth


def _zero(N, K):
    return np.zeros((N, K), np.int8), np.zeros((N, K // 128), np.uint16)


def test_sizes_of_a_ragged_matrix():
    # N = 40 -> NG = 2 groups of 32, K = 384 -> 3 blocks: codes 2 * 3 * 1 KB, scales 3 * 64 * 2 B
    assert layout.ternary_lut_sizes(40, 384) == [6144, 384]
    offs, total = layout.sections(layout.ternary_lut_sizes(40, 384))
    assert offs == [0, 6144] and total == 6144 + 512


def test_hand_placed_code_and_scale():
    """q[33][2*128 + 4*5 + 2] = -1 and scale(33, 2) = 1.0 in a 40 x 384 matrix.

    Row 33: group 1, lane 1. Column group c = 5 of block 2 sits at position
    t = (5 - 33) mod 32 = 4 (first half). Record (2, 1) starts at (2*2 + 1) * 1024
    = 5120; position 4 of lane 1 is 5120 + 1*16 + 4 = 5140. Column 2 of the group
    is at bits 4-5, code 10 -> byte 0x20. The scale is element 2*64 + 33 = 161 of
    section 1 (offset 6144): bytes 6466, 6467 = 00 3C.
    """
    q, s = _zero(40, 384)
    q[33, 2 * 128 + 4 * 5 + 2] = -1
    s[33, 2] = 0x3C00
    buf = np.frombuffer(ternary.pack_lut(q, s), np.uint8)
    nz = np.flatnonzero(buf)
    assert list(nz) == [5140, 6467]
    assert buf[5140] == 0x20 and buf[6466] == 0x00 and buf[6467] == 0x3C


def test_rotation_of_row_zero_and_row_31():
    """Row 0 keeps its groups in order; row 31 starts with group 31, then 0, 1, ..."""
    q, s = _zero(32, 128)
    for c in range(32):
        q[0, 4 * c] = 1                       # byte value 0x01 for every group of row 0
        q[31, 4 * c + 3] = -1 if c == 31 else 0
    q[31, 4 * 0 + 1] = 1                      # group 0 of row 31: column 1 -> 0x04
    buf = np.frombuffer(ternary.pack_lut(q, s), np.uint8)
    row0 = [buf[(t // 16) * 512 + 0 * 16 + t % 16] for t in range(32)]
    assert row0 == [1] * 32
    # row 31 (lane 31): position t holds group (t + 31) % 32: t = 0 -> group 31, t = 1 -> group 0
    assert buf[0 * 512 + 31 * 16 + 0] == 0x80            # column 3 of group 31: code 10 at bits 6-7
    assert buf[0 * 512 + 31 * 16 + 1] == 0x04            # column 1 of group 0: code 01 at bits 2-3


@pytest.mark.parametrize("N,K", [(1, 128), (31, 256), (33, 384), (70, 1152)])
def test_round_trip_and_same_codes_as_the_record_layout(N, K):
    w = synth.student_t4(synth.rng(N * 7 + K), (N, K))
    w[0, :128] = 0.0
    q, _, s16 = ternary.quantize(w)
    buf = ternary.pack_lut(q, s16)
    q2, s2 = ternary.unpack_lut(buf, N, K)
    q3, s3 = ternary.unpack(ternary.pack(q, s16), N, K)
    assert np.array_equal(q2, q) and np.array_equal(s2, s16)
    assert np.array_equal(q2, q3) and np.array_equal(s2, s3)
    # padding rows of the last group carry zero codes and zero scales
    offs, total = layout.sections(layout.ternary_lut_sizes(N, K))
    raw = np.frombuffer(buf, np.uint8)
    for n in range(N, layout.lut_groups(N) * 32):
        for b in range(K // 128):
            assert all(raw[offs[0] + layout.lut_byte_offset(n, b, t, N)] == 0 for t in range(32))


def test_unpack_rejects_code_11():
    q, s = _zero(2, 128)
    buf = bytearray(ternary.pack_lut(q, s))
    buf[layout.lut_byte_offset(1, 0, 7, 2)] = 0x0C      # code 11 at bits 2-3
    with pytest.raises(ValueError):
        ternary.unpack_lut(bytes(buf), 2, 128)


# ----------------------------------------------------------------------------- INT4 lookup layout

def test_int4_lut_sizes_of_a_ragged_matrix():
    # N = 40 -> NG = 2 groups of 32, K = 384 -> 3 blocks: codes 2 * 3 * 2 KB, scales 3 * 64 * 2 B
    assert layout.int4_lut_sizes(40, 384) == [12288, 384]
    offs, total = layout.sections(layout.int4_lut_sizes(40, 384))
    assert offs == [0, 12288] and total == 12288 + 512


def test_int4_lut_hand_placed_pair_and_scale():
    """q[33][2*128 + 80] = 5, q[33][2*128 + 81] = -3 and scale(33, 2) = 1.0 in a 40 x 384 matrix.

    Row 33: group 1, lane 1. Pair p = 40 of block 2 lies in the second half, at position
    t = 32 + (40 - 32 - 33) mod 32 = 39. Record (2, 1) starts at (2*2 + 1) * 2048 = 10240;
    position 39 of lane 1 is 10240 + (39 // 16)*512 + 1*16 + 39 % 16 = 11287. Column 80 is the
    low nibble (5), column 81 the high nibble (-3 = 0xD): byte 0xD5. The scale is element
    2*64 + 33 = 161 of section 1 (offset 12288): bytes 12610, 12611 = 00 3C.
    """
    from oracle import int4
    q = np.zeros((40, 384), np.int8)
    s = np.zeros((40, 3), np.uint16)
    q[33, 2 * 128 + 80], q[33, 2 * 128 + 81] = 5, -3
    s[33, 2] = 0x3C00
    buf = np.frombuffer(int4.pack_lut(q, s), np.uint8)
    nz = np.nonzero(buf)[0]
    assert list(nz) == [11287, 12611]
    assert buf[11287] == 0xD5 and buf[12610] == 0x00 and buf[12611] == 0x3C


def test_int4_lut_rotation_of_rows_0_and_31():
    """Pair 0 of row 0 sits at position 0 (offset 0); pair 0 of row 31 at position
    (0 - 31) mod 32 = 1, offset 31*16 + 1 = 497; pair 32 of row 31 at position
    32 + 1 = 33, offset (33 // 16)*512 + 31*16 + 1 = 1521. 7 and -7 pack as 0x97."""
    from oracle import int4
    q = np.zeros((32, 128), np.int8)
    s = np.zeros((32, 1), np.uint16)
    q[0, 0], q[0, 1] = 7, -7
    q[31, 0], q[31, 1] = 7, -7
    q[31, 64], q[31, 65] = 7, -7
    buf = np.frombuffer(int4.pack_lut(q, s), np.uint8)
    assert list(np.nonzero(buf)[0]) == [0, 497, 1521]
    assert buf[0] == buf[497] == buf[1521] == 0x97


def test_int4_lut_same_codes_as_the_record_layout_and_zero_padding():
    from oracle import int4
    w = synth.student_t4(synth.rng(12), (45, 640))
    q, _, s16 = int4.quantize(w)
    lut = int4.pack_lut(q, s16)
    q2, s2 = int4.unpack_lut(lut, 45, 640)
    q3, s3 = int4.unpack(int4.pack(q, s16), 45, 640)
    assert np.array_equal(q2, q3) and np.array_equal(s2, s3) and np.array_equal(q2, q)
    # rows 45..63 of the last group hold zero codes and zero scales
    raw = np.frombuffer(lut, np.uint8)
    offs, _ = layout.sections(layout.int4_lut_sizes(45, 640))
    for n in range(45, 64):
        for b in range(5):
            for t in range(64):
                assert raw[offs[0] + layout.lut4_byte_offset(n, b, t, 45)] == 0
            assert raw[offs[1] + 2 * layout.lut_scale_index(n, b, 45)] == 0
