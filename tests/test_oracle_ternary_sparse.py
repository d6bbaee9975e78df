"""Pins of the flagged sparse ternary oracle: hand-placed tiles, the all-zero-block scale
of 1.0, lossless round trip, and the page's bit accounting."""
import json
import os

import numpy as np

from conftest import GOLDEN
from oracle import layout, ternary, ternary_sparse as ts
from oracle.matvec import matvec
from quantized_gemv_unpack_gb300 import synth


def _hand_case():
    """N = 20 (groups: rows 0-15, rows 16-19 + 12 padding rows), K = 384 (blocks 0, 1, 2).
    Zero: tile (0, 1) (rows 0-15 of block 1) and tile (1, 0) (rows 16-19 of block 0; padding
    rows count as zero). Tile (1, 2) holds a single nonzero weight (row 19) and is stored."""
    w = synth.student_t4(synth.rng(21), (20, 384))
    w[0:16, 128:256] = 0.0
    w[16:20, 0:128] = 0.0
    w[16:19, 256:384] = 0.0
    w[19, 256:384] = 0.0
    w[19, 300] = 0.05
    return w


def test_hand_tiles():
    q, s16 = ts.quantize(_hand_case())
    stored = ts.tile_stored(q)
    assert stored.tolist() == [[True, False, True], [False, True, True]]
    buf, meta = ts.pack(q, s16)
    o = meta["offsets"]
    assert meta["T"] == 4
    assert np.frombuffer(buf, "<u4", 2, o[0]).tolist() == [0b101, 0b110]        # tile bitmaps
    assert np.frombuffer(buf, "<u4", 3, o[1]).tolist() == [0, 2, 4]             # tile starts
    assert np.frombuffer(buf, "<u2", 4, o[2]).tolist() == [0, 2, 1, 2]          # tile blocks
    # the lone weight of tile (1, 2) is q = +1 at row 19, column 300 = block 2, column 44:
    # record 0 of group 1 holds tiles (blocks 1, 2), row 3 of the group, tile 1, word 44 // 16 = 2
    codes = np.frombuffer(buf, "<u4", 4 * 128, o[3])
    word = codes[2 * 128 + (3 * 2 + 1) * 8 + 2]
    assert word == np.uint32(1) << np.uint32(layout.ternary_bit_pos(44))
    # all-zero blocks store the scale 1.0: row 19 block 0 (zero tile, not stored) and
    # rows 16-18 block 2 (inside the stored tile)
    scales = np.frombuffer(buf, "<u2", 4 * 16, o[4]).reshape(4, 16)
    assert scales[3, 0:3].tolist() == [0x3C00] * 3 and scales[3, 3] not in (0, 0x3C00)
    assert np.all(scales[3, 4:] == 0)                                           # padding rows


def test_zero_block_scale_is_one_where_dense_stores_zero():
    w = np.zeros((2, 256), np.float32)
    w[0, :128] = synth.student_t4(synth.rng(3), (1, 128))
    _, _, s16_dense = ternary.quantize(w)
    _, s16 = ts.quantize(w)
    assert s16_dense[0, 1] == 0 and s16[0, 1] == 0x3C00 and s16[1].tolist() == [0x3C00, 0x3C00]
    assert s16[0, 0] == s16_dense[0, 0]


def test_round_trip_and_matvec_equal_dense():
    g = synth.rng(22)
    w = synth.student_t4(g, (70, 1152))
    zero = g.random((5, 9)) < 0.3                              # drop about 30 % of the tiles
    for gi, b in zip(*np.nonzero(zero)):
        w[16 * gi:16 * gi + 16, 128 * b:128 * b + 128] = 0.0
    q, s16 = ts.quantize(w)
    buf, meta = ts.pack(q, s16)
    q2, s2 = ts.unpack(buf, meta)
    assert np.array_equal(q2, q) and np.array_equal(s2, s16)
    qd, _, sd = ternary.quantize(w)
    x = synth.activations_bf16(g, (3, 1152))
    from oracle.numerics import bf16_bits_to_f64
    xf = bf16_bits_to_f64(x)
    assert np.array_equal(matvec(ternary.dequant(q2, s2), xf), matvec(ternary.dequant(qd, sd), xf))
    assert meta["T"] == int((~ts.tile_stored(q)).size - (~ts.tile_stored(q)).sum())


def test_bit_accounting_reaches_the_pages_figure():
    """About 1.78 bits per parameter ("Ternary Bonsai 2", 1.1: 6 GB for 27B) with 2.125-bit
    blocks needs (1 - z) * 2.125 ~ 1.78, i.e. z ~ 16 % of the tiles left out; the index (mostly
    a 16-bit block number per stored tile of 2048 weights) costs about 0.008 bits per weight."""
    bpw = json.load(open(os.path.join(GOLDEN, "bits_per_weight.json")))
    target = 8 * bpw["bonsai_accounting"]["bytes"] / bpw["bonsai_accounting"]["params"]
    N, K = 4096, 4096
    G, KB = N // 16, K // 128
    T = int(round(G * KB * (1 - 0.165)))
    got = ts.bits_per_weight(N, K, T)
    assert abs(got - target) < 0.01
    assert 0.007 < got - (T / (G * KB)) * 2.125 < 0.009
