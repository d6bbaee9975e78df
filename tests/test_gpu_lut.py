"""GPU parity of the byte-lookup ternary layout (QMV_TERNARY2_LUT) and its matvec.

The GPU packer must write the oracle's bytes; qmv_unpack must give the oracle's
codes and scales; the lookup matvec (M = 1) must satisfy the library bound
|y - y_ref| <= 2e-3 * sum_k |w_hat_k x_k| on every row. Its tables and sums are
fp32 (exact products of the codes with bf16 activations, a handful of fp32
additions per table entry and one per code byte), so it is also held to
1e-5 * sum_k |w_hat_k x_k|, far below the contract, which a wrong column, sign
or scale would break.
"""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

RTOL = 2e-3
FP32_TOL = 1e-5


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_gemv_unpack_gb300 as q
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return q, torch, torch.device("cuda:0")


def _dev_bf16(torch, bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def _pack(q, torch, dev, w):
    N, K = w.shape
    d = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, N, K)
    p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
    q.qmv_pack_ternary(d, w if isinstance(w, torch.Tensor) else torch.from_numpy(w).to(dev), p)
    return d, p


def _check(y, yr, B, what, tol=FP32_TOL):
    err = np.abs(np.asarray(y, np.float64) - yr)
    worst = float((err / np.maximum(B, 1e-300)).max())
    assert np.all(err <= RTOL * B), f"{what}: outside the library bound, worst |err|/B = {worst:.3e}"
    assert np.all(err <= tol * B + 1e-37), f"{what}: worst |err|/B = {worst:.3e} above the fp32 path's {tol}"


@pytest.mark.parametrize("N,K", [(1, 128), (31, 384), (33, 256), (200, 1152), (64, 4096)])
def test_lut_packer_is_bit_exact(env, N, K):
    q, torch, dev = env
    from oracle import ternary
    from quantized_gemv_unpack_gb300 import synth
    w = synth.student_t4(synth.rng(N * 53 + K), (N, K))
    w[0, :128] = 0.0
    d, p = _pack(q, torch, dev, w)
    qq, _, s16 = ternary.quantize(w)
    assert np.array_equal(p.cpu().numpy(), np.frombuffer(ternary.pack_lut(qq, s16), np.uint8))
    qd = torch.empty((N, K), dtype=torch.int8, device=dev)
    sd = torch.empty((N, K // 128), dtype=torch.int16, device=dev)
    q.qmv_unpack(d, p, qd, sd)
    assert q.qmv_check_status() == 0
    assert np.array_equal(qd.cpu().numpy(), qq)
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), s16)


@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (33, 256), (200, 1152), (96, 5120), (40, 13824),
                                 (2500, 640), (3000, 1024), (4096, 4096)])
def test_lut_matvec_matches_oracle(env, N, K):
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(7000 + N + K)
    w = synth.student_t4(g, (N, K))
    xb = synth.activations_bf16(g, (1, K))
    d, p = _pack(q, torch, dev, w)
    y = torch.full((1, N), float("nan"), device=dev)
    q.qmv_run_ternary(d, p, _dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ternary.quantize(w)
    yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
    _check(y.cpu().numpy(), yr, B, f"N={N} K={K}")
    # the same call again gives the same bits (no atomics, fixed summation order)
    y2 = torch.empty_like(y)
    q.qmv_run_ternary(d, p, _dev_bf16(torch, xb, dev), y2)
    assert torch.equal(y, y2)


def test_lut_activation_range(env):
    """Tiny and huge activations (the whole bf16 range the fp32 tables can hold)."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(71)
    w = synth.student_t4(g, (96, 1024))
    d, p = _pack(q, torch, dev, w)
    qq, _, s16 = ternary.quantize(w)
    for scale in [1e-30, 1e-6, 1e4, 1e30]:
        xb = synth.to_bf16_bits(g.standard_normal((1, 1024)).astype(np.float32) * np.float32(scale))
        y = torch.empty((1, 96), device=dev)
        q.qmv_run_ternary(d, p, _dev_bf16(torch, xb, dev), y)
        yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
        _check(y.cpu().numpy(), yr, B, f"x scale {scale}")


def test_lut_sparse_codes(env):
    """One nonzero code per block against N(0,1) activations: a block's sum |w_hat x| is then a
    single term. The lookup path adds table entries that hold only the products of nonzero codes,
    so its error stays relative to that term (fp32 bound), unlike seeded fp16 chains."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    N, K = 96, 5120
    g = synth.rng(4243)
    w = np.zeros((N, K), np.float32)
    hit = g.integers(0, 128, size=(N, K // 128)) + 128 * np.arange(K // 128)[None, :]
    w[np.arange(N)[:, None], hit] = np.float32(0.02) * np.where(g.random((N, K // 128)) < 0.5, -1, 1)
    xb = synth.activations_bf16(g, (1, K))
    d, p = _pack(q, torch, dev, w)
    y = torch.full((1, N), float("nan"), device=dev)
    q.qmv_run_ternary(d, p, _dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ternary.quantize(w)
    assert np.all((qq != 0).reshape(N, K // 128, 128).sum(axis=2) == 1)
    yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
    _check(y.cpu().numpy(), yr, B, "sparse codes")


@pytest.mark.parametrize("kind", ["channels", "huge", "range"])
@pytest.mark.parametrize("K", [4096, 25600])
def test_lut_activation_outliers(env, kind, K):
    """Outlier channels (1000x, or one at 2^24) on columns whose codes are 0 in half of the rows,
    and a 2^24 range of magnitudes inside one row, at the full K of the stack (5120 / 25600) and
    of the single 4096 x 4096 matrix: zero codes add exactly 0 to a table entry, so the fp32
    bound holds."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    N = 96
    w, xb = synth.outlier_case(kind, N, K, 1, seed=K + 5)
    d, p = _pack(q, torch, dev, w)
    y = torch.full((1, N), float("nan"), device=dev)
    q.qmv_run_ternary(d, p, _dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = ternary.quantize(w)
    yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
    _check(y.cpu().numpy(), yr, B, f"{kind} K={K}")


def test_lut_invalid_byte_contributes_zero(env):
    """A code byte holding a code 11 adds nothing (its four columns count as 0); qmv_unpack flags it."""
    q, torch, dev = env
    from oracle import layout, ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(72)
    N, K = 40, 384
    w = synth.student_t4(g, (N, K))
    xb = synth.activations_bf16(g, (1, K))
    d, p = _pack(q, torch, dev, w)
    n, b, t = 33, 2, 4                                  # position 4 of row 33, block 2: column group 5
    p[layout.lut_byte_offset(n, b, t, N)] = 0xC3        # codes 11 at bits 0-1 and 6-7
    y = torch.empty((1, N), device=dev)
    q.qmv_run_ternary(d, p, _dev_bf16(torch, xb, dev), y)
    qq, _, s16 = ternary.quantize(w)
    c = (t + n) % 32
    qq[n, b * 128 + 4 * c: b * 128 + 4 * c + 4] = 0
    yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
    _check(y.cpu().numpy(), yr, B, "invalid byte")
    qd = torch.empty((N, K), dtype=torch.int8, device=dev)
    q.qmv_unpack(d, p, qd)
    assert q.qmv_check_status() == q.QMV_ERR_CORRUPT


def test_lut_many_tasks_one_launch(env):
    """400 matvecs of 1536 x 1024 in one launch (enough units for one CTA per unit, no cluster
    split), each with its own x; sampled rows of every task against the oracle."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(11, dev)
    N, K, T = 1536, 1024, 400
    mats, ws, xs, ys = [], [], [], []
    for i in range(T):
        w = synth.student_t4_torch(gen, (N, K), device=dev)
        mats.append(_pack(q, torch, dev, w))
        ws.append(w if i % 50 == 0 else None)
        xs.append(synth.activations_bf16_torch(gen, (1, K), device=dev))
        ys.append(torch.full((1, N), float("nan"), device=dev))
    batch = q.Batch(q.QMV_TERNARY2_LUT, [(d, p, x, y) for (d, p), x, y in zip(mats, xs, ys)], 1)
    batch.run()
    assert q.qmv_check_status() == 0
    assert all(bool(torch.isfinite(y).all()) for y in ys)
    # a second launch of the same batch writes the same bits (no atomics, fixed order)
    first = [y.clone() for y in ys]
    for y in ys:
        y.fill_(float("nan"))
    batch.run()
    assert all(torch.equal(a, y) for a, y in zip(first, ys))
    rng = np.random.default_rng(5)
    for i in range(0, T, 50):
        rows = np.unique(np.concatenate(([0, N - 1], rng.choice(N, 40, replace=False))))
        idx = torch.from_numpy(rows).to(dev)
        qq, _, s16 = ternary.quantize(ws[i][idx].cpu().numpy())
        xb = xs[i].view(torch.int16).cpu().numpy().view(np.uint16)
        yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
        _check(ys[i][:, idx].cpu().numpy(), yr, B, f"task {i}")


def test_lut_stack_layer_sampled(env):
    """One layer of the 27B-shaped stack (q, k, v, o, gate, up, down; hidden 5120, 40/8 heads of
    128, SwiGLU 25600) in one launch, as the benchmark runs it; sampled rows against the oracle."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(4, dev)
    H, I = 5120, 25600
    shapes = [("q", H, H), ("k", 1024, H), ("v", 1024, H), ("o", H, H), ("gate", I, H), ("up", I, H),
              ("down", H, I)]
    xs = {H: synth.activations_bf16_torch(gen, (1, H), device=dev),
          I: synth.activations_bf16_torch(gen, (1, I), device=dev)}
    rng = np.random.default_rng(4)
    tasks, checks = [], []
    for name, N, K in shapes:
        w = synth.student_t4_torch(gen, (N, K), device=dev)
        d, p = _pack(q, torch, dev, w)
        y = torch.full((1, N), float("nan"), device=dev)
        tasks.append((d, p, xs[K], y))
        rows = np.unique(np.concatenate(([0, N - 1], rng.choice(N, 24, replace=False))))
        idx = torch.from_numpy(rows).to(dev)
        checks.append((name, K, idx, w[idx].cpu().numpy(), y))
        del w
    q.qmv_run_batch(q.QMV_TERNARY2_LUT, tasks, 1)
    assert q.qmv_check_status() == 0
    for name, K, idx, wr, y in checks:
        qq, _, s16 = ternary.quantize(wr)
        xb = xs[K].view(torch.int16).cpu().numpy().view(np.uint16)
        yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
        _check(y[:, idx].cpu().numpy(), yr, B, name)


def test_lut_more_units_than_the_schedule_holds(env):
    """448 matvecs of 20480 x 128 give 4480 units of 2048 rows, more than the launch
    parameters list, so units go round-robin to the CTAs; sampled rows of every 32nd task
    against the oracle, and every output written."""
    q, torch, dev = env
    from oracle import ternary
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(12, dev)
    N, K, T = 20480, 128, q.QMV_MAX_BATCH
    tasks, keep = [], {}
    for i in range(T):
        w = synth.student_t4_torch(gen, (N, K), device=dev)
        d, p = _pack(q, torch, dev, w)
        x = synth.activations_bf16_torch(gen, (1, K), device=dev)
        y = torch.full((1, N), float("nan"), device=dev)
        tasks.append((d, p, x, y))
        if i % 32 == 0 or i == T - 1:
            keep[i] = w
        del w
    q.qmv_run_batch(q.QMV_TERNARY2_LUT, tasks, 1)
    assert q.qmv_check_status() == 0
    assert all(bool(torch.isfinite(t[3]).all()) for t in tasks)
    rng = np.random.default_rng(6)
    for i, w in keep.items():
        rows = np.unique(np.concatenate(([0, N - 1], rng.choice(N, 32, replace=False))))
        idx = torch.from_numpy(rows).to(dev)
        qq, _, s16 = ternary.quantize(w[idx].cpu().numpy())
        xb = tasks[i][2].view(torch.int16).cpu().numpy().view(np.uint16)
        yr, B = matvec_bf16x(ternary.dequant(qq, s16), xb)
        _check(tasks[i][3][:, idx].cpu().numpy(), yr, B, f"task {i}")


# ----------------------------------------------------------------------------- INT4 lookup layout

def _pack4(q, torch, dev, w):
    N, K = w.shape
    d = q.qmv_pack_desc(q.QMV_INT4_LUT, N, K)
    p = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
    q.qmv_pack_int4(d, w if isinstance(w, torch.Tensor) else torch.from_numpy(w).to(dev), p)
    return d, p


@pytest.mark.parametrize("N,K", [(1, 128), (31, 384), (33, 256), (200, 1152), (64, 4096)])
def test_int4_lut_packer_is_bit_exact(env, N, K):
    q, torch, dev = env
    from oracle import int4
    from quantized_gemv_unpack_gb300 import synth
    w = synth.student_t4(synth.rng(N * 17 + K), (N, K))
    w[0, :128] = 0.0
    d, p = _pack4(q, torch, dev, w)
    qq, _, s16 = int4.quantize(w)
    assert np.array_equal(p.cpu().numpy(), np.frombuffer(int4.pack_lut(qq, s16), np.uint8))
    qd = torch.empty((N, K), dtype=torch.int8, device=dev)
    sd = torch.empty((N, K // 128), dtype=torch.int16, device=dev)
    q.qmv_unpack(d, p, qd, sd)
    assert q.qmv_check_status() == 0
    assert np.array_equal(qd.cpu().numpy(), qq)
    assert np.array_equal(sd.cpu().numpy().view(np.uint16), s16)


@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (33, 256), (200, 1152), (96, 5120), (40, 13824), (4096, 4096)])
def test_int4_lut_matvec_matches_oracle(env, N, K):
    q, torch, dev = env
    from oracle import int4
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(7 * N + K)
    w = synth.student_t4(g, (N, K))
    xb = synth.activations_bf16(g, (1, K))
    d, p = _pack4(q, torch, dev, w)
    y = torch.full((1, N), float("nan"), device=dev)
    q.qmv_run_int4(d, p, _dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = int4.quantize(w)
    yr, B = matvec_bf16x(int4.dequant(qq, s16), xb)
    _check(y.cpu().numpy(), yr, B, f"int4 lut N={N} K={K}")


@pytest.mark.parametrize("case", ["saturated", "one_code", "channels", "huge", "range"])
def test_int4_lut_hard_inputs(env, case):
    """Saturated groups (every code at +-7 against activations just under a power of two), one
    nonzero code per group, outlier channels on zero codes and a 2^24 range inside one row, at
    K = 13824 (the INT4 layer set's down projection)."""
    q, torch, dev = env
    from oracle import int4
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    N, K = 96, 13824
    if case == "saturated":
        w = synth.student_t4(synth.rng(3), (N, K))
        w[0], w[1] = 0.02, -0.02
        w[2, 0::2], w[2, 1::2] = 0.02, -0.02
        xb = synth.to_bf16_bits(np.full((1, K), 0.99, np.float32))
    elif case == "one_code":
        g = synth.rng(4)
        w = np.zeros((N, K), np.float32)
        hit = g.integers(0, 128, size=(N, K // 128)) + 128 * np.arange(K // 128)[None, :]
        w[np.arange(N)[:, None], hit] = np.float32(0.02) * np.where(g.random((N, K // 128)) < 0.5, -1, 1)
        xb = synth.activations_bf16(g, (1, K))
    else:
        w, xb = synth.outlier_case(case, N, K, 1, seed=K + 9)
    d, p = _pack4(q, torch, dev, w)
    y = torch.full((1, N), float("nan"), device=dev)
    q.qmv_run_int4(d, p, _dev_bf16(torch, xb, dev), y)
    assert q.qmv_check_status() == 0
    qq, _, s16 = int4.quantize(w)
    yr, B = matvec_bf16x(int4.dequant(qq, s16), xb)
    _check(y.cpu().numpy(), yr, B, f"int4 lut {case}")


def test_int4_lut_layer_set_batched_sampled(env):
    """The INT4 GQA layer set (hidden 5120, 40/8 heads, SwiGLU 13824) in the lookup layout, one
    batched launch as the benchmark runs it, and each matrix alone (a smaller launch, whose blocks
    a cluster may split differently); sampled rows of both against the oracle."""
    q, torch, dev = env
    from oracle import int4
    from oracle.matvec import matvec_bf16x
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(1, dev)
    shapes = synth.gqa_layer_shapes(5120, 40, 8, 128, 13824)
    mats, ws = [], []
    for name, N, K in shapes:
        w = synth.student_t4_torch(gen, (N, K), device=dev)
        mats.append(_pack4(q, torch, dev, w))
        ws.append(w)
    xs = {K: synth.activations_bf16_torch(gen, (1, K), device=dev) for K in {5120, 13824}}
    ys = [torch.empty((1, N), device=dev) for _, N, _ in shapes]
    q.qmv_run_batch(q.QMV_INT4_LUT, [(d, p, xs[K], y) for (d, p), (_, N, K), y in zip(mats, shapes, ys)], 1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    for (d, p), (name, N, K), w, y in zip(mats, shapes, ws, ys):
        y1 = torch.empty_like(y)
        q.qmv_run_int4(d, p, xs[K], y1)
        rows = np.unique(np.concatenate(([0, N - 1], rng.choice(N, 24, replace=False))))
        qq, _, s16 = int4.quantize(w[torch.from_numpy(rows).to(dev)].cpu().numpy())
        xb = xs[K].view(torch.int16).cpu().numpy().view(np.uint16)
        yr, B = matvec_bf16x(int4.dequant(qq, s16), xb)
        idx = torch.from_numpy(rows).to(dev)
        _check(y[:, idx].cpu().numpy(), yr, B, name)
        _check(y1[:, idx].cpu().numpy(), yr, B, name + " alone")
    assert q.qmv_check_status() == 0


def test_int4_lut_rejects_mixed_batches_and_m_above_1(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    w = synth.student_t4(synth.rng(2), (32, 256))
    d4, p4 = _pack4(q, torch, dev, w)
    dt, pt = _pack(q, torch, dev, w)
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((2, 32), device=dev)
    with pytest.raises(q.QmvError):
        q.qmv_run_int4(d4, p4, x, y)                                   # M = 2
    with pytest.raises(q.QmvError):
        q.qmv_run_batch(q.QMV_INT4_LUT, [(d4, p4, x[:1], y[:1]), (dt, pt, x[:1], y[1:])], 1)
