"""GPU parity of the Cassandra-2 (MX shared-exponent) draft and target paths (through the C ABI).

Materialised draft and target weights must equal the oracle's bit for bit, and the
fused matvecs must satisfy |y - y_ref| <= 2e-3 * sum_k |w_k x_k| against the oracle's
decoded weights.
"""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

RTOL = 2e-3


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_gemv_unpack_gb300 as q
    assert torch.cuda.is_available()
    return q, torch, torch.device("cuda:0")


def _dev(torch, a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _bf16(torch, bits, dev):
    return _dev(torch, bits.view(np.int16), dev).view(torch.bfloat16)


def _run(q, torch, dev, W, X, M, seed):
    from quantized_gemv_unpack_gb300 import synth
    N, K = W.shape
    d, buf = q.cass_mx_pack_host(W, X)
    packed = _dev(torch, buf, dev)
    xb = synth.activations_bf16(synth.rng(seed), (M, K))
    x = _bf16(torch, xb, dev)
    yd = torch.full((M, N), float("nan"), device=dev)
    yt = torch.full((M, N), float("nan"), device=dev)
    wd = torch.empty((N, K), dtype=torch.int16, device=dev)
    wt = torch.empty((N, K), dtype=torch.int16, device=dev)
    q.cass_decode_draft(d, packed, x, yd, wd)
    q.cass_reconstruct(d, packed, x, yt, wt)
    assert q.qmv_check_status() == 0
    u16 = lambda t: t.cpu().numpy().view(np.uint16)
    return xb, yd.cpu().numpy(), yt.cpu().numpy(), u16(wd), u16(wt)


@pytest.mark.parametrize("N,K,M", [(1, 64, 1), (24, 256, 1), (40, 512, 5), (33, 1024, 3), (7, 192, 2), (130, 4096, 8)])
def test_mx_draft_and_target_match_oracle(env, N, K, M):
    q, torch, dev = env
    from oracle import cassandra_mx as mx
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(N * 11 + K)
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, 64, K)
    xb, yd, yt, wd, wt = _run(q, torch, dev, W, X, M, N + M + 1)
    ref, meta = mx.pack(W, X)
    draft, target = mx.draft(ref, meta), mx.reconstruct(ref, meta)
    assert np.array_equal(wd, draft)
    assert np.array_equal(wt, target)
    for y, wbits in [(yd, draft), (yt, target)]:
        yr, B = matvec_bf16x(bf16_bits_to_f64(wbits), xb)
        assert np.all(np.abs(y - yr) <= RTOL * B)


def test_mx_special_values(env):
    """All 65,536 bf16 patterns (zeros, subnormals, exponent 255) through both paths, bit for bit."""
    q, torch, dev = env
    from oracle import cassandra_mx as mx
    from quantized_gemv_unpack_gb300 import synth
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    W = allp.reshape(1024, 64)
    X = synth.to_bf16_bits(np.ones((2, 64), np.float32))
    d, buf = q.cass_mx_pack_host(W, X)
    packed = _dev(torch, buf, dev)
    x = _bf16(torch, synth.to_bf16_bits(np.zeros((1, 64), np.float32)), dev)
    wd = torch.empty((1024, 64), dtype=torch.int16, device=dev)
    wt = torch.empty((1024, 64), dtype=torch.int16, device=dev)
    q.cass_decode_draft(d, packed, x, None, wd)
    q.cass_reconstruct(d, packed, x, None, wt)
    assert q.qmv_check_status() == 0
    ref, meta = mx.pack(W, X)
    assert np.array_equal(wd.cpu().numpy().view(np.uint16), mx.draft(ref, meta))
    assert np.array_equal(wt.cpu().numpy().view(np.uint16), mx.reconstruct(ref, meta))


@pytest.mark.parametrize("K", [256, 512])
@pytest.mark.parametrize("M", [1, 3])
def test_mx_rows_with_full_bitmap_words(env, M, K):
    """A row pruning a whole 32-column word and one keeping one: bit-exact weights, y in tolerance."""
    q, torch, dev = env
    from oracle import cassandra_mx as mx
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(44)
    w = synth.student_t4(g, (24, K))
    w[0, 0:32] = 1e-7
    w[1, 32:64] = 1.0
    W = synth.to_bf16_bits(w)
    X = synth.to_bf16_bits(np.ones((8, K), np.float32))
    ref, meta = mx.pack(W, X)
    d, buf = q.cass_mx_pack_host(W, X)
    packed = torch.from_numpy(buf).to(dev)
    xb = synth.activations_bf16(synth.rng(45), (M, K))
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    yd = torch.empty((M, 24), device=dev)
    yt = torch.empty((M, 24), device=dev)
    wd = torch.empty((24, K), dtype=torch.int16, device=dev)
    wt = torch.empty((24, K), dtype=torch.int16, device=dev)
    q.cass_decode_draft(d, packed, x, yd, wd)
    q.cass_reconstruct(d, packed, x, yt, wt)
    assert q.qmv_check_status() == 0
    draft, target = mx.draft(ref, meta), mx.reconstruct(ref, meta)
    assert np.array_equal(wd.cpu().numpy().view(np.uint16), draft)
    assert np.array_equal(wt.cpu().numpy().view(np.uint16), target)
    for y, Wr in ((yd, draft), (yt, target)):
        yr, B = matvec_bf16x(bf16_bits_to_f64(Wr), xb)
        assert np.all(np.abs(y.cpu().numpy() - yr) <= RTOL * B)


def test_mx_full_mlp_matrix_sampled(env):
    """The 14336 x 4096 MLP matrix of the Cassandra workload: target weights of sampled rows
    bit-exact, matvec of sampled rows within the bound."""
    q, torch, dev = env
    from oracle import cassandra_mx as mx
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(2)
    N, K = 14336, 4096
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, 128, K)
    xb, yd, yt, wd, wt = _run(q, torch, dev, W, X, 5, 3)
    rows = np.unique(np.concatenate(([0, N - 1], np.random.default_rng(0).choice(N, 40, replace=False))))
    ref, meta = mx.pack(W[rows], X)
    assert np.array_equal(wt[rows], mx.reconstruct(ref, meta))
    assert np.array_equal(wd[rows], mx.draft(ref, meta))
    yr, B = matvec_bf16x(bf16_bits_to_f64(mx.reconstruct(ref, meta)), xb)
    assert np.all(np.abs(yt[:, rows] - yr) <= RTOL * B)
