"""The library's flagged sparse ternary packer (host) against the oracle's: byte-identical buffers."""
import numpy as np
import pytest

import quantized_gemv_unpack_gb300 as q
from oracle import ternary, ternary_sparse as ts
from quantized_gemv_unpack_gb300 import build, synth


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _weights(N, K, frac, seed):
    g = synth.rng(seed)
    w = synth.student_t4(g, (N, K))
    G = (N + 15) // 16
    zero = g.random((G, K // 128)) < frac
    for gi, b in zip(*np.nonzero(zero)):
        w[16 * gi:16 * gi + 16, 128 * b:128 * b + 128] = 0.0
    return w


@pytest.mark.parametrize("N,K,frac", [(1, 128, 0.0), (20, 384, 0.3), (70, 1152, 0.17), (64, 4096, 0.5), (33, 1024, 1.0)])
def test_sparse_packer_matches_oracle(N, K, frac):
    w = _weights(N, K, frac, N + K)
    qd, _, sd = ternary.quantize(w)
    dense = q.qmv_pack_desc(q.QMV_TERNARY2, N, K)
    d, out = q.qmv_sparse_pack_host(dense, np.frombuffer(ternary.pack(qd, sd), np.uint8))
    qs, ss = ts.quantize(w)
    ref, meta = ts.pack(qs, ss)
    assert d.format == q.QMV_TERNARY2_SPARSE and d.n_symbols == meta["T"]
    assert [d.off[i] for i in range(5)] == meta["offsets"] and [d.bytes[i] for i in range(5)] == meta["sizes"]
    assert np.array_equal(out, np.frombuffer(ref, np.uint8))


def test_sparse_packer_rejects_bad_input():
    import ctypes
    dense = q.qmv_pack_desc(q.QMV_TERNARY2, 16, 256)
    buf = np.zeros(dense.total_bytes, np.uint8)
    d = q.qmv_desc()
    L = q.lib()
    assert L.qmv_sparse_pack_host(None, buf.ctypes.data, ctypes.byref(d), None, 0) == q.QMV_ERR_ARG
    assert L.qmv_sparse_pack_host(ctypes.byref(dense), None, ctypes.byref(d), None, 0) == q.QMV_ERR_ARG
    assert L.qmv_sparse_pack_host(ctypes.byref(dense), buf.ctypes.data, ctypes.byref(d), None, 0) == 0
    assert d.n_symbols == 0                                  # all-zero matrix: nothing stored
    small = np.zeros(8, np.uint8)
    assert L.qmv_sparse_pack_host(ctypes.byref(dense), buf.ctypes.data, ctypes.byref(d), small.ctypes.data, 8) == q.QMV_ERR_ARG
