"""Packed-weight files on the host (no GPU): CRC-32, write / open / read round trip, and
corruption caught by the per-section, table and header CRCs ("Ternary Bonsai 2" 3.6: the
packed model is exported as a file that inference loads)."""
import os
import zlib

import numpy as np
import pytest


@pytest.fixture(scope="module")
def q():
    from quantized_gemv_unpack_gb300 import build
    build.build()
    import quantized_gemv_unpack_gb300 as q
    return q


def test_crc32_check_value_and_zlib(q):
    # the catalogue check value of CRC-32 (reflected 0xEDB88320, init and final xor ~0)
    assert q.qmv_crc32(b"123456789") == 0xCBF43926
    assert q.qmv_crc32(b"") == 0
    g = np.random.default_rng(1)
    data = g.integers(0, 256, size=100003, dtype=np.uint8)
    for lo, hi in [(0, 1), (3, 20), (1, 100003), (7, 4096 + 5)]:
        piece = np.ascontiguousarray(data[lo:hi])
        assert q.qmv_crc32(piece) == zlib.crc32(piece.tobytes())
    # continuation: crc(a + b) from crc(a)
    a, b = data[:1001], data[1001:5000]
    assert q.qmv_crc32(np.ascontiguousarray(b), q.qmv_crc32(a)) == zlib.crc32(data[:5000].tobytes())


def _items(q):
    g = np.random.default_rng(7)
    items = []
    for name, fmt, N, K in [("layer0.q", q.QMV_TERNARY2, 200, 1152), ("layer0.o", q.QMV_INT4, 33, 384),
                            ("layer0.down", q.QMV_TERNARY2_LUT, 70, 640)]:
        d = q.qmv_pack_desc(fmt, N, K)
        items.append((name, d, g.integers(0, 256, size=d.total_bytes, dtype=np.uint8)))
    return items


def test_file_round_trip(q, tmp_path):
    items = _items(q)
    path = str(tmp_path / "m.qmv")
    q.qmv_file_write(path, items)
    assert os.path.getsize(path) % 4096 == 0
    with q.QmvFile(path) as f:
        assert len(f) == len(items)
        for i, (name, d, buf) in enumerate(items):
            nm, dd = f.tensor(i)
            assert nm == name
            assert (dd.format, dd.N, dd.K, dd.total_bytes) == (d.format, d.N, d.K, d.total_bytes)
            assert dd.sections() == d.sections()
            assert f.find(name) == i
            out = np.zeros(d.total_bytes, np.uint8)
            f.read_host(i, out)
            assert np.array_equal(out, buf)
        with pytest.raises(q.QmvError):
            f.find("absent")
        with pytest.raises(q.QmvError):
            f.read_host(0, np.zeros(10, np.uint8))          # capacity below total_bytes


def test_cassandra_descriptor_round_trip(q, tmp_path):
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(3)
    W = synth.to_bf16_bits(synth.student_t4(g, (24, 256)))
    X, _ = synth.calibration_bf16(g, 16, 256)
    d, buf = q.cass_pack_host(W, X)
    path = str(tmp_path / "c.qmv")
    q.qmv_file_write(path, [("mlp.up", d, buf)])
    with q.QmvFile(path) as f:
        _, dd = f.tensor(0)
        assert dd.n_symbols == d.n_symbols and dd.sections() == d.sections()
        out = np.zeros(d.total_bytes, np.uint8)
        f.read_host(0, out)
        assert np.array_equal(out, buf)


def _flip(path, offset):
    with open(path, "r+b") as fh:
        fh.seek(offset)
        b = fh.read(1)
        fh.seek(offset)
        fh.write(bytes([b[0] ^ 0x10]))


def test_flipped_data_byte_is_caught_per_section(q, tmp_path):
    items = _items(q)
    path = str(tmp_path / "m.qmv")
    q.qmv_file_write(path, items)
    with q.QmvFile(path) as f:
        off1 = f.tensor(1)[1]
    # tensor 1 starts at the second 4096-aligned data offset; flip a byte inside its scale section
    with open(path, "rb") as fh:
        hdr = fh.read(64)
    data0 = int.from_bytes(hdr[24:32], "little")
    t0 = items[0][1].total_bytes
    start1 = data0 + (t0 + 4095) // 4096 * 4096
    _flip(path, start1 + off1.off[1] + 5)
    with q.QmvFile(path) as f:
        f.read_host(0, np.zeros(items[0][1].total_bytes, np.uint8))   # other tensors still load
        with pytest.raises(q.QmvError) as e:
            f.read_host(1, np.zeros(items[1][1].total_bytes, np.uint8))
        assert e.value.status == q.QMV_ERR_CORRUPT


@pytest.mark.parametrize("where", ["magic", "header", "table", "truncate"])
def test_damaged_header_or_table_is_rejected(q, tmp_path, where):
    items = _items(q)
    path = str(tmp_path / "m.qmv")
    q.qmv_file_write(path, items)
    if where == "magic":
        _flip(path, 0)
    elif where == "header":
        _flip(path, 9)                                        # n_tensors
    elif where == "table":
        _flip(path, 64 + 70)                                  # inside entry 0's descriptor
    else:
        with open(path, "r+b") as fh:
            fh.truncate(os.path.getsize(path) - 4096)
    with pytest.raises(q.QmvError) as e:
        q.QmvFile(path)
    assert e.value.status == q.QMV_ERR_CORRUPT


def test_write_rejects_bad_input(q, tmp_path):
    items = _items(q)
    with pytest.raises(q.QmvError):
        q.qmv_file_write(str(tmp_path / "d.qmv"), [items[0], (items[0][0], items[1][1], items[1][2])])  # same name
    with pytest.raises(q.QmvError):
        q.qmv_file_write(str(tmp_path / "l.qmv"), [("x" * 64, items[0][1], items[0][2])])   # name too long
