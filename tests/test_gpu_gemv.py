"""GPU parity of the ternary and INT4 paths against the float64 oracle (through the C ABI).

Packed bytes and decoded codes must be bit-identical to the oracle's; matvec
outputs of both kernels (fp16-FMA and tensor-core, forced through
qmv_desc.flags) must satisfy |y - y_ref| <= 2e-3 * sum_k |w_hat_k x_k| for every
row, including blocks of identical codes, one nonzero code per block, outlier
activation channels on zero codes and a 2^24 range of activations in one row.
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
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return q, torch, torch.device("cuda:0")


FORMATS = {}


def _fmt(q, name):
    from oracle import int4, ternary
    if name == "ternary":
        return q.QMV_TERNARY2, ternary, q.qmv_pack_ternary, q.qmv_run_ternary
    return q.QMV_INT4, int4, q.qmv_pack_int4, q.qmv_run_int4


def _to_dev_bf16(torch, bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


PATHS = {"fma": 1, "mma": 2}   # QMV_FLAG_PATH_FMA / QMV_FLAG_PATH_MMA


def _pack(q, torch, dev, name, w, path=None):
    fmt, ref, pack, run = _fmt(q, name)
    N, K = w.shape
    d = q.qmv_pack_desc(fmt, N, K)
    d.flags = PATHS[path] if path else 0
    packed = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
    pack(d, torch.from_numpy(w).to(dev), packed)
    return d, packed


def _check_bound(y, yr, B, what):
    err = np.abs(y.astype(np.float64) - yr)
    worst = float((err / np.maximum(B, 1e-300)).max())
    assert np.all(err <= RTOL * B), f"{what}: worst |err|/B = {worst:.3e}"
    return worst


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (33, 256), (200, 1152), (64, 13824), (4096, 4096)])
def test_packer_is_bit_exact(env, name, N, K):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, _ = _fmt(q, name)
    w = synth.student_t4(synth.rng(N * 131 + K), (N, K))
    w[0, :128] = 0.0                                   # an all-zero block
    d, packed = _pack(q, torch, dev, name, w)
    qq, _, s16 = ref.quantize(w)
    assert np.array_equal(packed.cpu().numpy(), np.frombuffer(ref.pack(qq, s16), np.uint8))
    # decode on the GPU: int8 codes and scales identical to the oracle's
    qd = torch.empty((N, K), dtype=torch.int8, device=dev)
    sd = torch.empty((N, K // 128), dtype=torch.int16, device=dev)
    q.qmv_unpack(d, packed, qd, sd)
    assert q.qmv_check_status() == 0
    assert np.array_equal(qd.cpu().numpy(), qq)
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), s16)


def test_unpack_flags_invalid_ternary_code(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    w = synth.student_t4(synth.rng(5), (4, 256))
    d, packed = _pack(q, torch, dev, "ternary", w)
    packed[5] = 0xFF                                   # codes 11 in word 1 of row 0
    qd = torch.empty((4, 256), dtype=torch.int8, device=dev)
    q.qmv_unpack(d, packed, qd)
    assert q.qmv_check_status() == q.QMV_ERR_CORRUPT
    assert q.qmv_check_status() == 0                   # the word is cleared after reading


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (33, 256), (200, 1152), (96, 5120), (40, 13824)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("path", ["fma", "mma"])
def test_matvec_matches_oracle(env, name, N, K, M, path):
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, run = _fmt(q, name)
    g = synth.rng(1000 * M + N + K)
    w = synth.student_t4(g, (N, K))
    xb = synth.activations_bf16(g, (M, K))
    d, packed = _pack(q, torch, dev, name, w, path)
    y = torch.full((M, N), float("nan"), device=dev)
    run(d, packed, _to_dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ref.quantize(w)
    yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
    _check_bound(y.cpu().numpy(), yr, B, f"{name} N={N} K={K} M={M} {path}")


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("path", ["fma", "mma"])
def test_saturated_blocks_stay_finite(env, name, M, path):
    """Constant rows (every code at its extreme) against constant activations just under a power
    of two: the fp16 chains of the fp16-FMA kernel are largest here (they must not overflow), and
    all their roundings point the same way. Each chain of four exact products rounds three times
    (at most 3 * 2^-11 of its sum of |terms|), so both kernels stay within 2e-3."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, run = _fmt(q, name)
    N, K = 48, 1024
    w = synth.student_t4(synth.rng(77), (N, K))
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
    xb = synth.to_bf16_bits(x)
    d, packed = _pack(q, torch, dev, name, w, path)
    y = torch.full((M, N), float("nan"), device=dev)
    run(d, packed, _to_dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ref.quantize(w)
    yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
    yy = y.cpu().numpy()
    assert np.all(np.isfinite(yy))
    _check_bound(yy, yr, B, f"{name} saturated M={M} {path}")


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("path", ["fma", "mma"])
def test_sparse_codes_stay_within_bound(env, name, M, path):
    """One nonzero code per block against N(0,1) activations: the bound's sum |w_hat x| of a block
    is a single term, so any leak of the zero codes' activations into the sums (an offset such as
    1 + q/2 that is subtracted again) shows up here. Both kernels decode zero codes to an exact 0."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, run = _fmt(q, name)
    N, K = 64, 5120
    g = synth.rng(4242 + M)
    w = np.zeros((N, K), np.float32)
    hit = g.integers(0, 128, size=(N, K // 128)) + 128 * np.arange(K // 128)[None, :]
    w[np.arange(N)[:, None], hit] = np.float32(0.02) * np.where(g.random((N, K // 128)) < 0.5, -1, 1)
    xb = synth.activations_bf16(g, (M, K))
    d, packed = _pack(q, torch, dev, name, w, path)
    y = torch.full((M, N), float("nan"), device=dev)
    run(d, packed, _to_dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ref.quantize(w)
    nz = (qq != 0).reshape(N, K // 128, 128).sum(axis=2)
    assert np.all(nz == 1), "every block holds exactly one nonzero code"
    yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
    _check_bound(y.cpu().numpy(), yr, B, f"{name} sparse codes M={M} {path}")


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("kind", ["channels", "huge", "range"])  # synth.OUTLIER_KINDS
@pytest.mark.parametrize("M", [1, 2, 8])
@pytest.mark.parametrize("path", ["fma", "mma"])
def test_activation_outliers_stay_within_bound(env, name, kind, M, path):
    """Massive activation channels on columns whose codes are 0 in half of the rows, and a 2^24
    range of magnitudes inside one row, at the full K of the configurations (4096, 13824)."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, run = _fmt(q, name)
    for K in (4096, 13824):
        N = 96
        w, xb = synth.outlier_case(kind, N, K, M, seed=K + M)
        d, packed = _pack(q, torch, dev, name, w, path)
        y = torch.full((M, N), float("nan"), device=dev)
        run(d, packed, _to_dev_bf16(torch, xb, dev), y)
        assert q.qmv_check_status() == 0
        qq, _, s16 = ref.quantize(w)
        yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
        _check_bound(y.cpu().numpy(), yr, B, f"{name} {kind} K={K} M={M} {path}")


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("M", [1, 8])
def test_cfg_ternary_4096_square_full(env, name, M):
    """The single-matrix workload (4096 x 4096) at batch 1 and as a verification of
    1 + 7 draft tokens (M = 8, tensor-core kernel), every row against the oracle."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, run = _fmt(q, name)
    g = synth.rng(0)
    w = synth.student_t4(g, (4096, 4096))
    xb = synth.activations_bf16(g, (M, 4096))
    d, packed = _pack(q, torch, dev, name, w)
    y = torch.empty((M, 4096), device=dev)
    run(d, packed, _to_dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ref.quantize(w)
    yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
    _check_bound(y.cpu().numpy(), yr, B, f"{name} 4096x4096 M={M}")


@pytest.mark.parametrize("path", ["fma", "mma"])
def test_activation_range_is_handled(env, path):
    """Tiny and huge activations (bf16 range far outside fp16's) stay within the bound."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from oracle import ternary
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(77)
    w = synth.student_t4(g, (64, 1024))
    d, packed = _pack(q, torch, dev, "ternary", w, path)
    qq, _, s16 = ternary.quantize(w)
    for scale in [1e-30, 1e-6, 1e4, 1e30]:
        x = synth.to_bf16_bits(g.standard_normal((2, 1024)).astype(np.float32) * np.float32(scale))
        y = torch.empty((2, 64), device=dev)
        q.qmv_run_ternary(d, packed, _to_dev_bf16(torch, x, dev), y)
        yr, B = matvec_bf16x(ternary.dequant(qq, s16), x)
        _check_bound(y.cpu().numpy(), yr, B, f"x scale {scale}")


@pytest.mark.parametrize("path", ["fma", "mma"])
def test_strided_activations_and_outputs(env, path):
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from oracle import int4
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(78)
    N, K, M = 48, 640, 3
    w = synth.student_t4(g, (N, K))
    xb = synth.activations_bf16(g, (M, K))
    d, packed = _pack(q, torch, dev, "int4", w, path)
    xbig = torch.zeros((M, K + 64), dtype=torch.bfloat16, device=dev)
    xbig[:, :K] = _to_dev_bf16(torch, xb, dev)
    ybig = torch.full((M, N + 12), 7.0, device=dev)
    q.qmv_run_int4(d, packed, xbig, ybig)
    qq, _, s16 = int4.quantize(w)
    yr, B = matvec_bf16x(int4.dequant(qq, s16), xb)
    yy = ybig.cpu().numpy()
    _check_bound(yy[:, :N], yr, B, "strided")
    assert (yy[:, N:] == 7.0).all()                     # nothing written past N


@pytest.mark.parametrize("name", ["ternary", "int4"])
@pytest.mark.parametrize("M", [1, 2, 6])
def test_batch_equals_separate_calls(env, name, M):
    """q|k|v sharing one x in a single launch give the same bits as separate launches,
    on the fp16-FMA kernel (ternary, M = 1) and the tensor-core kernel (INT4, and M >= 2)."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    fmt, ref, _, run = _fmt(q, name)
    g = synth.rng(90)
    K = 1280
    shapes = [(320, K), (64, K), (64, K), (96, 2560)]
    ws = [synth.student_t4(g, s) for s in shapes]
    mats = [_pack(q, torch, dev, name, w) for w in ws]
    xb1 = synth.activations_bf16(g, (M, K))
    xb2 = synth.activations_bf16(g, (M, 2560))
    x1, x2 = _to_dev_bf16(torch, xb1, dev), _to_dev_bf16(torch, xb2, dev)
    xs, xbs = [x1, x1, x1, x2], [xb1, xb1, xb1, xb2]
    ys_b = [torch.empty((M, s[0]), device=dev) for s in shapes]
    q.qmv_run_batch(fmt, [(d, p, x, y) for (d, p), x, y in zip(mats, xs, ys_b)], M)
    for (d, p), x, xb, w, yb in zip(mats, xs, xbs, ws, ys_b):
        y = torch.empty_like(yb)
        run(d, p, x, y)
        assert torch.equal(y, yb)   # both kernels add partial sums in a fixed order
        qq, _, s16 = ref.quantize(w)
        yr, B = matvec_bf16x(ref.dequant(qq, s16), xb)
        _check_bound(yb.cpu().numpy(), yr, B, "batched")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_int4_gqa_layer_set_sampled(env, M):
    """The INT4 GQA layer set (hidden 5120, 40/8 heads of 128, SwiGLU 13824) at full size, one batched
    launch as the benchmark runs it; sampled rows of every matrix against the oracle."""
    q, torch, dev = env
    from oracle import int4
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(1, dev)
    shapes = synth.gqa_layer_shapes(5120, 40, 8, 128, 13824)
    mats, ws = [], []
    for name, N, K in shapes:
        w = synth.student_t4_torch(gen, (N, K), device=dev)
        d = q.qmv_pack_desc(q.QMV_INT4, N, K)
        p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
        q.qmv_pack_int4(d, w, p)
        mats.append((d, p))
        ws.append(w)
    xs = {K: synth.activations_bf16_torch(gen, (M, K), device=dev) for K in {5120, 13824}}
    ys = [torch.empty((M, N), device=dev) for _, N, _ in shapes]
    q.qmv_run_batch(q.QMV_INT4, [(d, p, xs[K], y) for (d, p), (_, N, K), y in zip(mats, shapes, ys)], M)
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    for (d, p), (name, N, K), w, y in zip(mats, shapes, ws, ys):
        rows = np.unique(np.concatenate(([0, N - 1], rng.choice(N, 24, replace=False))))
        wr = w[torch.from_numpy(rows).to(dev)].cpu().numpy()
        qq, _, s16 = int4.quantize(wr)
        # decoded codes and scales of the sampled rows are the oracle's
        qd = torch.empty((N, K), dtype=torch.int8, device=dev)
        sd = torch.empty((N, K // 128), dtype=torch.int16, device=dev)
        q.qmv_unpack(d, p, qd, sd)
        idx = torch.from_numpy(rows).to(dev)
        assert np.array_equal(qd[idx].cpu().numpy(), qq), name
        assert np.array_equal(sd[idx].cpu().numpy().view(np.uint16), s16), name
        xb = xs[K].view(torch.int16).cpu().numpy().view(np.uint16)
        yr, B = matvec_bf16x(int4.dequant(qq, s16), xb)
        _check_bound(y[:, torch.from_numpy(rows).to(dev)].cpu().numpy(), yr, B, f"{name} M={M}")


@pytest.mark.parametrize("path", ["fma", "mma"])
def test_smaller_launch_does_not_break_a_larger_one(env, path):
    """A launch needing less shared memory between two larger ones of the same kernel
    (the per-kernel shared-memory limit must only ever grow)."""
    q, torch, dev = env
    from oracle.matvec import matvec_bf16x
    from oracle import int4
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(91)
    M = 4
    runs = []
    for K in (13824, 384, 13824):
        w = synth.student_t4(g, (24, K))
        xb = synth.activations_bf16(g, (M, K))
        d, packed = _pack(q, torch, dev, "int4", w, path)
        y = torch.empty((M, 24), device=dev)
        q.qmv_run_int4(d, packed, _to_dev_bf16(torch, xb, dev), y)
        runs.append((w, xb, y))
    assert q.qmv_check_status() == 0
    for w, xb, y in runs:
        qq, _, s16 = int4.quantize(w)
        yr, B = matvec_bf16x(int4.dequant(qq, s16), xb)
        _check_bound(y.cpu().numpy(), yr, B, f"K={w.shape[1]}")


@pytest.mark.parametrize("path", ["fma", "mma"])
def test_bounded_wait_timeout_is_reported(env, path):
    """QMV_FLAG_TEST_WAIT_TIMEOUT makes the kernel's first wait one that nothing completes (1 ms
    limit): the call returns, y is left unwritten, qmv_check_status reports QMV_ERR_TIMEOUT once,
    and the next clean call on the same context gives 0 and the oracle's result."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(606)
    N, K, M = 64, 2048, 1
    w = synth.student_t4(g, (N, K))
    xb = synth.activations_bf16(g, (M, K))
    d, packed = _pack(q, torch, dev, "ternary", w, path)
    x = _to_dev_bf16(torch, xb, dev)
    d.flags |= q.QMV_FLAG_TEST_WAIT_TIMEOUT
    y = torch.full((M, N), float("nan"), device=dev)
    q.qmv_run_ternary(d, packed, x, y)
    code = q.qmv_check_status()
    assert code == q.QMV_ERR_TIMEOUT
    assert torch.isnan(y).all()                          # the kernel gave up before writing
    assert q.qmv_check_status() == 0                     # the word was cleared
    d.flags &= ~q.QMV_FLAG_TEST_WAIT_TIMEOUT
    q.qmv_run_ternary(d, packed, x, y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ternary.quantize(w)
    yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
    _check_bound(y.cpu().numpy(), yr, B, f"after timeout {path}")


def test_unknown_flag_bits_are_rejected(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    w = synth.student_t4(synth.rng(607), (16, 256))
    d, packed = _pack(q, torch, dev, "int4", w)
    d.flags = 0x40
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((1, 16), device=dev)
    with pytest.raises(q.QmvError):
        q.qmv_run_int4(d, packed, x, y)
