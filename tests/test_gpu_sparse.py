"""GPU parity of the flagged sparse ternary matvec (through the C ABI) against the oracle:
|y - y_ref| <= 2e-3 * sum_k |w_hat_k x_k| for every row, with tiles left out."""
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


def _weights(N, K, frac, seed):
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(seed)
    w = synth.student_t4(g, (N, K))
    G = (N + 15) // 16
    zero = g.random((G, K // 128)) < frac
    for gi, b in zip(*np.nonzero(zero)):
        w[16 * gi:16 * gi + 16, 128 * b:128 * b + 128] = 0.0
    return w


def _pack_sparse(q, torch, dev, w):
    """Dense pack on the GPU, sparse pack on the host from its copy, upload."""
    N, K = w.shape
    dense = q.qmv_pack_desc(q.QMV_TERNARY2, N, K)
    p = torch.empty(dense.total_bytes, dtype=torch.uint8, device=dev)
    q.qmv_pack_ternary(dense, torch.from_numpy(w).to(dev), p)
    d, host = q.qmv_sparse_pack_host(dense, p.cpu().numpy())
    return d, torch.from_numpy(host).to(dev)


@pytest.mark.parametrize("N,K,frac", [(1, 128, 0.0), (20, 384, 0.3), (70, 1152, 0.17), (200, 4096, 0.5), (33, 1024, 1.0)])
@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_sparse_matvec_matches_oracle(env, N, K, frac, M):
    q, torch, dev = env
    from oracle import ternary, ternary_sparse as ts
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    w = _weights(N, K, frac, 1000 * M + N + K)
    d, packed = _pack_sparse(q, torch, dev, w)
    xb = synth.activations_bf16(synth.rng(M + N), (M, K))
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.full((M, N), float("nan"), device=dev)
    q.qmv_run_ternary(d, packed, x, y)
    assert q.qmv_check_status() == 0
    qs, ss = ts.quantize(w)
    yr, B = matvec_bf16x(ternary.dequant(qs, ss), xb)
    yy = y.cpu().numpy()
    assert np.all(np.abs(yy - yr) <= RTOL * B), f"worst {np.max(np.abs(yy - yr) / np.maximum(B, 1e-300)):.3e}"


def _run_sparse(q, torch, dev, w, xb):
    from oracle import ternary, ternary_sparse as ts
    from oracle.matvec import matvec_bf16x
    M, N = xb.shape[0], w.shape[0]
    d, packed = _pack_sparse(q, torch, dev, w)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.full((M, N), float("nan"), device=dev)
    q.qmv_run_ternary(d, packed, x, y)
    assert q.qmv_check_status() == 0
    qs, ss = ts.quantize(w)
    yr, B = matvec_bf16x(ternary.dequant(qs, ss), xb)
    return y.cpu().numpy(), yr, B


def _check(yy, yr, B, what):
    err = np.abs(yy.astype(np.float64) - yr)
    assert np.all(err <= RTOL * B), f"{what}: worst |err|/B = {np.max(err / np.maximum(B, 1e-300)):.3e}"


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_sparse_saturated_blocks(env, M):
    """Identical codes against identical activations just under a power of two (the fp16 chains'
    roundings all point the same way), with zero tiles in between."""
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    N, K = 48, 1024
    w = _weights(N, K, 0.3, 77)
    w[0] = 0.02
    w[1] = -0.02
    w[2, : K // 2], w[2, K // 2:] = 0.02, -0.02
    w[3, 0::2], w[3, 1::2] = 0.02, -0.02
    x = np.full((M, K), 0.99, np.float32)
    if M > 1:
        x[1] = -0.99
    if M > 2:
        x[2, 0::2], x[2, 1::2] = 0.99, -0.99
        x[3] = np.float32(0.99) * np.sign(synth.rng(78).standard_normal(K)).astype(np.float32)
    yy, yr, B = _run_sparse(q, torch, dev, w, synth.to_bf16_bits(x))
    assert np.all(np.isfinite(yy))
    _check(yy, yr, B, f"saturated M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_sparse_one_code_per_block(env, M):
    """One nonzero code per block of the stored tiles: a zero code must add exactly nothing."""
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    N, K = 64, 5120
    g = synth.rng(4244 + M)
    w = np.zeros((N, K), np.float32)
    hit = g.integers(0, 128, size=(N, K // 128)) + 128 * np.arange(K // 128)[None, :]
    w[np.arange(N)[:, None], hit] = np.float32(0.02) * np.where(g.random((N, K // 128)) < 0.5, -1, 1)
    w[16:32, 128 * 5:128 * 9] = 0.0                     # a few zero tiles
    yy, yr, B = _run_sparse(q, torch, dev, w, synth.activations_bf16(g, (M, K)))
    _check(yy, yr, B, f"one code per block M={M}")


@pytest.mark.parametrize("kind", ["channels", "huge", "range"])
@pytest.mark.parametrize("M", [1, 2, 8])
def test_sparse_activation_outliers(env, kind, M):
    """Outlier channels on columns whose codes are 0 in half of the rows, and a 2^24 range of
    magnitudes inside one row, at K = 13824 (the longest K whose activations fit shared memory in
    one piece at M <= 4) and K = 5120 at M = 8."""
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    N, K = 96, (13824 if M <= 4 else 5120)
    w, xb = synth.outlier_case(kind, N, K, M, seed=31 + M)
    g = synth.rng(32)
    zero = g.random(((N + 15) // 16, K // 128)) < 0.2
    for gi, b in zip(*np.nonzero(zero)):
        w[16 * gi:16 * gi + 16, 128 * b:128 * b + 128] = 0.0
    yy, yr, B = _run_sparse(q, torch, dev, w, xb)
    _check(yy, yr, B, f"{kind} M={M}")


def test_sparse_batch_equals_separate_calls(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    shapes = [(320, 1280, 0.2), (64, 1280, 0.0), (96, 2560, 0.4)]
    mats = [_pack_sparse(q, torch, dev, _weights(N, K, f, 7 + i)) for i, (N, K, f) in enumerate(shapes)]
    g = synth.rng(9)
    xs = {K: torch.from_numpy(synth.activations_bf16(g, (1, K)).view(np.int16)).to(dev).view(torch.bfloat16)
          for K in (1280, 2560)}
    ys = [torch.empty((1, N), device=dev) for N, _, _ in shapes]
    q.qmv_run_batch(q.QMV_TERNARY2_SPARSE, [(d, p, xs[K], y) for (d, p), (_, K, _), y in zip(mats, shapes, ys)], 1)
    for (d, p), (N, K, _), yb in zip(mats, shapes, ys):
        y = torch.empty_like(yb)
        q.qmv_run_ternary(d, p, xs[K], y)
        assert torch.equal(y, yb)
    assert q.qmv_check_status() == 0


def test_sparse_corrupt_block_index_is_reported(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    w = _weights(32, 512, 0.2, 5)
    d, packed = _pack_sparse(q, torch, dev, w)
    bad = packed.clone()
    bad[d.off[2]:d.off[2] + 2] = torch.tensor([0xFF, 0x7F], dtype=torch.uint8, device=dev)   # block 32767
    x = torch.from_numpy(synth.activations_bf16(synth.rng(1), (1, 512)).view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((1, 32), device=dev)
    q.qmv_run_ternary(d, bad, x, y)
    assert q.qmv_check_status() == q.QMV_ERR_CORRUPT
    assert q.qmv_check_status() == 0


def test_sparse_rejects_what_it_cannot_serve(env):
    q, torch, dev = env
    w = _weights(16, 128, 0.0, 3)
    d, packed = _pack_sparse(q, torch, dev, w)
    x = torch.zeros((9, 128), dtype=torch.bfloat16, device=dev)
    y = torch.empty((9, 16), device=dev)
    with pytest.raises(q.QmvError):                     # M = 9: the sparse path serves M <= 8
        q.qmv_run_ternary(d, packed, x, y)
