"""GPU parity of the online KV encoder (through the C ABI): byte-identical to the oracle,
losslessly decoded by the Cassandra target kernel, slot overflow reported."""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_gemv_unpack_gb300 as q
    assert torch.cuda.is_available()
    return q, torch, torch.device("cuda:0")


def _kv(T, D, seed, scale=0.5):
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(seed)
    v = g.standard_normal((T, D)).astype(np.float32) * np.float32(scale)
    v[:, :: max(1, D // 16)] *= 20                      # channel outliers, as keys have
    return synth.to_bf16_bits(v)


@pytest.mark.parametrize("T,D,slot", [(1, 32, 8), (7, 128, 16), (64, 1024, 96), (300, 512, 64)])
def test_encoder_matches_oracle_and_decodes_losslessly(env, T, D, slot):
    q, torch, dev = env
    from oracle import cassandra, cassandra_kv as kv
    from oracle.numerics import bf16_fields
    W = _kv(T, D, T + D)
    W[0, 1] = 0x7FC0                                     # a NaN and ties
    W[min(1, T - 1), 2:6] = W[min(1, T - 1), 6]
    cb = kv.codebook_from(bf16_fields(W[: max(1, T // 8)])[1])
    x = torch.from_numpy(W.view(np.int16)).to(dev)
    d = q.cass_kv_encode(x, cb, slot)
    packed = torch.full((d.total_bytes,), 0xAB, dtype=torch.uint8, device=dev)
    q.cass_kv_encode(x, cb, slot, packed)
    ref, meta, fits = kv.pack(W, cb, slot)
    assert fits.all()
    assert q.qmv_check_status() == 0
    assert d.total_bytes == meta["total"] and [d.off[i] for i in range(7)] == meta["offsets"]
    assert np.array_equal(packed.cpu().numpy(), np.frombuffer(ref, np.uint8))
    # the Cassandra target kernel rebuilds every original bit
    wt = torch.empty((T, D), dtype=torch.int16, device=dev)
    q.cass_reconstruct(d, packed, torch.zeros((1, D), dtype=torch.bfloat16, device=dev), None, wt)
    assert q.qmv_check_status() == 0
    assert np.array_equal(wt.cpu().numpy().view(np.uint16), W)
    assert np.array_equal(cassandra.reconstruct(ref, meta), W)


def test_encoder_slot_overflow_is_reported(env):
    q, torch, dev = env
    from oracle import cassandra_kv as kv
    W = np.full((2, 64), 0x3F80, np.uint16)
    W[1] = 0x3C00
    cb = kv.codebook_from(np.array([127]))
    x = torch.from_numpy(W.view(np.int16)).to(dev)
    d = q.cass_kv_encode(x, cb, 4)
    packed = torch.zeros(d.total_bytes, dtype=torch.uint8, device=dev)
    q.cass_kv_encode(x, cb, 4, packed)
    assert q.qmv_check_status() == q.QMV_ERR_UNSUPPORTED
    assert q.qmv_check_status() == 0
    ref, meta, fits = kv.pack(W, cb, 4)
    assert fits.tolist() == [True, False]
    assert np.array_equal(packed.cpu().numpy(), np.frombuffer(ref, np.uint8))   # the codes that fit
