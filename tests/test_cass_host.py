"""The library's host-side Cassandra packer against the oracle's (no GPU needed): byte-identical buffers."""
import numpy as np
import pytest

import quantized_gemv_unpack_gb300 as q
from oracle import cassandra as cs
from quantized_gemv_unpack_gb300 import build, synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _compare(W, X):
    d, out = q.cass_pack_host(W, X)
    ref, meta = cs.pack(W, X)
    assert d.total_bytes == meta["total"]
    assert [d.off[i] for i in range(7)] == meta["offsets"]
    assert [d.bytes[i] for i in range(7)] == meta["sizes"]
    assert d.n_symbols == meta["n_symbols"]
    assert d.format == q.QMV_CASS and d.N == W.shape[0] and d.K == W.shape[1]
    assert np.array_equal(out, np.frombuffer(ref, np.uint8))
    return d, out, meta


@pytest.mark.parametrize("N,K,R", [(1, 32, 1), (24, 256, 16), (40, 512, 128), (130, 1024, 128)])
def test_host_packer_matches_oracle(N, K, R):
    g = synth.rng(N + K + R)
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, R, K)
    _compare(W, X)


def test_host_packer_special_values_and_ties():
    # every bf16 pattern (zeros, subnormals, inf, NaN) in both roles, and exact score ties
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    X = synth.to_bf16_bits(np.ones((2, 32), np.float32))
    W = np.zeros((2048, 32), np.uint16)
    W.reshape(-1)[:] = allp
    _compare(W, X)
    Wt = np.full((4, 64), 0x3C00, np.uint16)          # all scores equal: lower columns kept
    _compare(Wt, synth.to_bf16_bits(np.ones((3, 64), np.float32)))


def test_host_packer_size_query_and_errors():
    g = synth.rng(5)
    W = synth.to_bf16_bits(synth.student_t4(g, (8, 64)))
    X, _ = synth.calibration_bf16(g, 4, 64)
    d = q.qmv_desc()
    import ctypes
    L = q.lib()
    assert L.cass_pack_host(W.ctypes.data, 8, 64, X.ctypes.data, 4, ctypes.byref(d), None, 0) == 0
    assert d.total_bytes > 0
    small = np.zeros(16, np.uint8)
    assert L.cass_pack_host(W.ctypes.data, 8, 64, X.ctypes.data, 4, ctypes.byref(d), small.ctypes.data, 16) == q.QMV_ERR_ARG
    assert L.cass_pack_host(W.ctypes.data, 8, 60, X.ctypes.data, 4, ctypes.byref(d), None, 0) == q.QMV_ERR_ARG
    assert L.cass_pack_host(None, 8, 64, X.ctypes.data, 4, ctypes.byref(d), None, 0) == q.QMV_ERR_ARG


# ----------------------------------------------------------------------------- Cassandra-2 (MX)

def _compare_mx(W, X):
    from oracle import cassandra_mx as mx
    d, out = q.cass_mx_pack_host(W, X)
    ref, meta = mx.pack(W, X)
    assert d.total_bytes == meta["total"] and d.format == q.QMV_CASS_MX and d.group == 32
    assert [d.off[i] for i in range(6)] == meta["offsets"]
    assert [d.bytes[i] for i in range(6)] == meta["sizes"]
    assert np.array_equal(out, np.frombuffer(ref, np.uint8))
    # the layout depends only on N and K
    d2 = q.qmv_pack_desc(q.QMV_CASS_MX, W.shape[0], W.shape[1], 32)
    assert [d2.off[i] for i in range(8)] == [d.off[i] for i in range(8)] and d2.total_bytes == d.total_bytes


@pytest.mark.parametrize("N,K,R", [(1, 64, 1), (24, 256, 16), (40, 512, 128), (130, 1024, 128)])
def test_mx_host_packer_matches_oracle(N, K, R):
    g = synth.rng(7 * N + K + R)
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, R, K)
    _compare_mx(W, X)


def test_mx_host_packer_special_values_and_ties():
    # every bf16 pattern (zeros, subnormals, exponent 255) in both roles, and exact score ties
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    X = synth.to_bf16_bits(np.ones((2, 64), np.float32))
    W = np.zeros((1024, 64), np.uint16)
    W.reshape(-1)[:] = allp
    _compare_mx(W, X)
    _compare_mx(np.full((4, 128), 0x3C00, np.uint16), synth.to_bf16_bits(np.ones((3, 128), np.float32)))


def test_mx_host_packer_errors():
    import ctypes
    g = synth.rng(6)
    W = synth.to_bf16_bits(synth.student_t4(g, (8, 128)))
    X, _ = synth.calibration_bf16(g, 4, 128)
    d = q.qmv_desc()
    L = q.lib()
    assert L.cass_mx_pack_host(W.ctypes.data, 8, 96, X.ctypes.data, 4, ctypes.byref(d), None, 0) == q.QMV_ERR_ARG
    small = np.zeros(16, np.uint8)
    assert L.cass_mx_pack_host(W.ctypes.data, 8, 128, X.ctypes.data, 4, ctypes.byref(d), small.ctypes.data, 16) == q.QMV_ERR_ARG
    with pytest.raises(q.QmvError):
        q.qmv_pack_desc(q.QMV_CASS_MX, 8, 128, 128)          # group must be 32
