"""GPU parity of the Cassandra draft and target paths (through the C ABI).

Materialised draft weights must equal the oracle's bit for bit, reconstructed
weights must equal the original bf16 bits (the lossless invariant), and the
fused matvecs must satisfy |y - y_ref| <= 2e-3 * sum_k |w_k x_k|.
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


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _run(q, torch, dev, W, X, M, seed):
    from quantized_gemv_unpack_gb300 import synth
    N, K = W.shape
    d, buf = q.cass_pack_host(W, X)
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
    return d, packed, xb, yd.cpu().numpy(), yt.cpu().numpy(), _u16(wd), _u16(wt)


@pytest.mark.parametrize("N,K,M", [(1, 32, 1), (24, 256, 1), (40, 512, 5), (33, 1024, 3), (7, 160, 2), (19, 96, 4), (130, 4096, 8)])
def test_draft_and_target_match_oracle(env, N, K, M):
    q, torch, dev = env
    from oracle import cassandra as cs
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(N * 7 + K)
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, 128, K)
    d, packed, xb, yd, yt, wd, wt = _run(q, torch, dev, W, X, M, N + M)
    ref, meta = cs.pack(W, X)
    assert np.array_equal(wd, cs.draft(ref, meta))
    assert np.array_equal(wt, W)
    for y, wbits in [(yd, cs.draft(ref, meta)), (yt, W)]:
        yr, B = matvec_bf16x(bf16_bits_to_f64(wbits), xb)
        assert np.all(np.abs(y - yr) <= RTOL * B)


def test_special_values_roundtrip(env):
    """All 65,536 bf16 patterns come back bit-exactly through the target path."""
    q, torch, dev = env
    from oracle import cassandra as cs
    from quantized_gemv_unpack_gb300 import synth
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    W = allp.reshape(2048, 32)
    X = synth.to_bf16_bits(np.ones((2, 32), np.float32))
    d, buf = q.cass_pack_host(W, X)
    packed = _dev(torch, buf, dev)
    x = _bf16(torch, synth.activations_bf16(synth.rng(1), (1, 32)), dev)
    wt = torch.empty((2048, 32), dtype=torch.int16, device=dev)
    wd = torch.empty((2048, 32), dtype=torch.int16, device=dev)
    q.cass_reconstruct(d, packed, x, None, wt)
    q.cass_decode_draft(d, packed, x, None, wd)
    assert q.qmv_check_status() == 0
    assert np.array_equal(_u16(wt), W)
    ref, meta = cs.pack(W, X)
    assert np.array_equal(_u16(wd), cs.draft(ref, meta))


def _edge_rows(K, seed):
    """Rows that defeat a one-word cursor step: row 0 prunes a whole 32-column word, row 1 keeps
    one, row 2 keeps values of 40 distinct exponents once each (unary codes of rank >= 32, so
    empty stream words), the other rows are ordinary."""
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(seed)
    w = synth.student_t4(g, (24, K))
    w[0, 0:32] = 1e-7
    w[1, 32:64] = 1.0
    w[2, :] = 1e-30
    w[2, 0:40] = [2.0 ** -e for e in range(1, 41)]
    w[2, 40:K // 2] = 0.75
    return synth.to_bf16_bits(w)


@pytest.mark.parametrize("K", [256, 512])
@pytest.mark.parametrize("M", [1, 3])
def test_rows_with_empty_words(env, M, K):
    """Full-word runs in the bitmap and empty exponent-stream words: bit-exact weights, y in tolerance."""
    q, torch, dev = env
    from oracle import cassandra as cs
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    W = _edge_rows(K, 41)
    X, _ = synth.calibration_bf16(synth.rng(42), 8, K)
    X[:] = synth.to_bf16_bits(np.ones(X.shape, np.float32))
    ref, meta = cs.pack(W, X)
    assert not meta["keep"][0, :32].any() and meta["keep"][1, 32:64].all()
    d, packed, xb, yd, yt, wd, wt = _run(q, torch, dev, W, X, M, 43)
    assert np.array_equal(wt, W) and np.array_equal(wd, cs.draft(ref, meta))
    for y, Wr in ((yd, cs.draft(ref, meta)), (yt, W)):
        yr, B = matvec_bf16x(bf16_bits_to_f64(Wr), xb)
        assert np.all(np.abs(y - yr) <= RTOL * B)


def test_mlp_matrix_full_size_sampled(env):
    """The 14336 x 4096 MLP matrix with 128 calibration rows (1% outlier channels x20): draft at M=1,
    target at M=5; reconstruction checked on every weight, draft weights and outputs on sampled rows."""
    q, torch, dev = env
    from oracle import cassandra as cs
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(2)
    N, K = 14336, 4096
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, chans = synth.calibration_bf16(g, 128, K)
    d, buf = q.cass_pack_host(W, X)
    packed = _dev(torch, buf, dev)
    x1 = synth.activations_bf16(g, (1, K))
    x5 = synth.activations_bf16(g, (5, K))
    yd = torch.empty((1, N), device=dev)
    yt = torch.empty((5, N), device=dev)
    wd = torch.empty((N, K), dtype=torch.int16, device=dev)
    wt = torch.empty((N, K), dtype=torch.int16, device=dev)
    q.cass_decode_draft(d, packed, _bf16(torch, x1, dev), yd, wd)
    q.cass_reconstruct(d, packed, _bf16(torch, x5, dev), yt, wt)
    assert q.qmv_check_status() == 0
    assert np.array_equal(_u16(wt), W)                          # lossless, every bit
    rows = np.unique(np.concatenate(([0, N - 1], np.random.default_rng(0).choice(N, 40, replace=False))))
    keep = cs.wanda_keep(W[rows], cs.column_norms(X))
    draft_ref = np.where(keep, W[rows] & np.uint16(0xFFF0), np.uint16(0))
    assert np.array_equal(_u16(wd)[rows], draft_ref)
    yr, B = matvec_bf16x(bf16_bits_to_f64(draft_ref), x1)
    assert np.all(np.abs(yd.cpu().numpy()[:, rows] - yr) <= RTOL * B)
    yr, B = matvec_bf16x(bf16_bits_to_f64(W[rows]), x5)
    assert np.all(np.abs(yt.cpu().numpy()[:, rows] - yr) <= RTOL * B)
    # the speculation data is what the draft reads: far smaller than the dense bf16 matrix
    spec = sum(d.bytes[i] for i in range(5))
    assert spec < 0.35 * N * K * 2


def test_corrupt_streams_are_reported(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(9)
    W = synth.to_bf16_bits(synth.student_t4(g, (16, 256)))
    X, _ = synth.calibration_bf16(g, 8, 256)
    d, buf = q.cass_pack_host(W, X)
    x = _bf16(torch, synth.activations_bf16(g, (1, 256)), dev)
    y = torch.empty((1, 16), device=dev)
    # no codeword ends in the exponent stream
    bad = buf.copy()
    bad[d.off[2]:d.off[2] + d.bytes[2]] = 0
    q.cass_decode_draft(d, _dev(torch, bad, dev), x, y)
    assert q.qmv_check_status() == q.QMV_ERR_CORRUPT
    # a bitmap row keeping every column
    bad = buf.copy()
    bad[d.off[0]:d.off[0] + 32] = 0xFF
    q.cass_reconstruct(d, _dev(torch, bad, dev), x, y)
    assert q.qmv_check_status() == q.QMV_ERR_CORRUPT
    # a unary rank past the codebook: a long run of zeros before the first one
    bad = buf.copy()
    bad[d.off[2]:d.off[2] + 64] = 0
    bad[d.off[2] + 64] = 1
    q.cass_decode_draft(d, _dev(torch, bad, dev), x, y)
    assert q.qmv_check_status() == q.QMV_ERR_CORRUPT
    # the untouched buffer is clean
    q.cass_decode_draft(d, _dev(torch, buf, dev), x, y)
    assert q.qmv_check_status() == 0


@pytest.mark.parametrize("mx", [False, True])
@pytest.mark.parametrize("n_draft", [1, 4, 7])
def test_speculate_step_draft_then_verify(env, mx, n_draft):
    """One self-speculative step ("Cassandra" 2, 3.2 figures b and c): n_draft draft matvecs at
    M = 1 from the speculation data, then one target pass at M = n_draft + 1. The draft outputs
    match the draft matvec of the oracle's draft weights, and the verification output matches
    the dense bf16 matvec of the original weights (Cassandra-1: lossless rebuild) or of the
    oracle's MX target values (Cassandra-2), each within the bound."""
    q, torch, dev = env
    from oracle import cassandra as cs
    from oracle import cassandra_mx as cmx
    from oracle.matvec import matvec_bf16x
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(900 + n_draft)
    N, K = 200, 1024
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, 128, K)
    d, buf = (q.cass_mx_pack_host if mx else q.cass_pack_host)(W, X)
    packed = _dev(torch, buf, dev)
    xb = synth.activations_bf16(g, (n_draft + 1, K))
    x = _bf16(torch, xb, dev)
    yd = torch.full((n_draft, N), float("nan"), device=dev)
    yt = torch.full((n_draft + 1, N), float("nan"), device=dev)
    q.cass_speculate_step(d, packed, x, yd, yt)
    assert q.qmv_check_status() == 0
    if mx:
        ref, meta = cmx.pack(W, X)
        w_draft, w_target = bf16_bits_to_f64(cmx.draft(ref, meta)), bf16_bits_to_f64(cmx.reconstruct(ref, meta))
    else:
        ref, meta = cs.pack(W, X)
        w_draft, w_target = bf16_bits_to_f64(cs.draft(ref, meta)), bf16_bits_to_f64(W)
    yr, B = matvec_bf16x(w_draft, xb[:n_draft])
    assert np.all(np.abs(yd.cpu().numpy() - yr) <= RTOL * B)
    yr, B = matvec_bf16x(w_target, xb)
    assert np.all(np.abs(yt.cpu().numpy() - yr) <= RTOL * B)


def test_speculate_step_rejects_bad_arguments(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(5)
    W = synth.to_bf16_bits(synth.student_t4(g, (16, 256)))
    X, _ = synth.calibration_bf16(g, 16, 256)
    d, buf = q.cass_pack_host(W, X)
    packed = _dev(torch, buf, dev)
    x = torch.zeros((9, 256), dtype=torch.bfloat16, device=dev)
    with pytest.raises(q.QmvError):                      # n_draft = 8 > 7
        q.cass_speculate_step(d, packed, x, torch.zeros((8, 16), device=dev), torch.zeros((9, 16), device=dev))
    y = torch.zeros((9, 16), device=dev)
    with pytest.raises(q.QmvError):                      # y_draft overlaps y_target
        q.cass_speculate_step(d, packed, x[:5], y[1:5], y[0:5])
