"""Every hot-path entry point issues only stream-ordered work (no synchronisation, no
allocation), so a decode loop can capture its calls in a CUDA graph and replay them. The
tests capture each call once, replay the graph on new inputs written into the captured
buffers, and compare with eager calls: bit for bit where the kernel's summation order is
fixed, within the method's bound where fp32 atomics set it (the MoE down phase)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_gemv_unpack_gb300 as q
    assert torch.cuda.is_available()
    return q, torch, torch.device("cuda:0")


def _replay_matches(torch, call, inputs, outputs, exact=True, rtol=None):
    """Capture call() on torch's capture stream, then for two new input draws: copy them
    into the captured buffers, replay, and compare every output with an eager call."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call()  # warm-up outside the capture (first-call lookups and attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    gen = torch.Generator(device=inputs[0].device).manual_seed(7)
    for _ in range(2):
        for t in inputs:
            if t.dtype == torch.bfloat16:
                t.copy_(torch.randn(t.shape, generator=gen, device=t.device).to(torch.bfloat16))
            else:
                t.copy_(torch.randn(t.shape, generator=gen, device=t.device))
        g.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in outputs]
        call()
        torch.cuda.synchronize()
        for a, b in zip(got, outputs):
            if exact:
                assert torch.equal(a, b)
            else:
                assert torch.allclose(a, b, rtol=rtol, atol=rtol * b.abs().max().item())


@pytest.mark.parametrize("fmt,M", [("ternary", 1), ("ternary", 4), ("ternary_lut", 1), ("int4", 1), ("int4", 8),
                                   ("int4_lut", 1)])
def test_matvec_in_a_graph(env, fmt, M):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    N, K = 1200, 3072
    gen = synth.torch_generator(11, dev)
    f = {"ternary": q.QMV_TERNARY2, "ternary_lut": q.QMV_TERNARY2_LUT, "int4": q.QMV_INT4, "int4_lut": q.QMV_INT4_LUT}[fmt]
    d = q.qmv_pack_desc(f, N, K)
    w = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
    pack = q.qmv_pack_int4 if fmt.startswith("int4") else q.qmv_pack_ternary
    run = q.qmv_run_int4 if fmt.startswith("int4") else q.qmv_run_ternary
    pack(d, synth.student_t4_torch(gen, (N, K), device=dev), w)
    x = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    y = torch.empty((M, N), device=dev)
    _replay_matches(torch, lambda: run(d, w, x, y), [x], [y])
    assert q.qmv_check_status() == 0


def test_batch_in_a_graph(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(12, dev)
    shapes = [(640, 1024), (2048, 1024), (1024, 3072)]
    tasks, xs, ys = [], [], []
    for N, K in shapes:
        d = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, N, K)
        w = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
        q.qmv_pack_ternary(d, synth.student_t4_torch(gen, (N, K), device=dev), w)
        x = torch.empty((1, K), dtype=torch.bfloat16, device=dev)
        y = torch.empty((1, N), device=dev)
        tasks.append((d, w, x, y))
        xs.append(x)
        ys.append(y)
    b = q.Batch(q.QMV_TERNARY2_LUT, tasks, 1)
    _replay_matches(torch, lambda: b.run(torch.cuda.current_stream()), xs, ys)
    assert q.qmv_check_status() == 0


def test_moe_in_a_graph(env):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    E, H, I, topk, M = 16, 512, 256, 4, 2
    gen = synth.torch_generator(13, dev)
    gu = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, 2 * I, H)
    dn = q.qmv_pack_desc(q.QMV_TERNARY2_LUT, H, I)
    stride = gu.total_bytes + dn.total_bytes
    buf = torch.empty(E * stride, dtype=torch.uint8, device=dev)
    for e in range(E):
        rec = buf[e * stride:(e + 1) * stride]
        q.qmv_pack_ternary(gu, synth.student_t4_torch(gen, (2 * I, H), device=dev), rec[:gu.total_bytes])
        q.qmv_pack_ternary(dn, synth.student_t4_torch(gen, (H, I), device=dev), rec[gu.total_bytes:])
    logits = torch.empty((M, E), device=dev)
    x = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((M, H), device=dev)
    ws = torch.zeros(q.moe_workspace_size(E, topk, M, H, I), dtype=torch.uint8, device=dev)
    call = lambda: q.moe_qmv_run(gu, dn, buf, stride, gu.total_bytes, E, logits, topk, x, y, ws,
                                 torch.cuda.current_stream())
    # the down phase adds into y by fp32 atomics: equal up to summation order
    _replay_matches(torch, call, [logits, x], [y], exact=False, rtol=1e-5)
    assert q.qmv_check_status() == 0


@pytest.mark.parametrize("what", ["draft", "reconstruct", "speculate"])
def test_cassandra_in_a_graph(env, what):
    q, torch, dev = env
    from quantized_gemv_unpack_gb300 import synth
    g = synth.rng(14)
    N, K = 256, 1024
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, _ = synth.calibration_bf16(g, 16, K)
    d, host = q.cass_pack_host(W, X)
    packed = torch.from_numpy(host).to(dev)
    if what == "speculate":
        x = torch.empty((5, K), dtype=torch.bfloat16, device=dev)
        yd = torch.empty((4, N), device=dev)
        yt = torch.empty((5, N), device=dev)
        call = lambda: q.cass_speculate_step(d, packed, x, yd, yt, torch.cuda.current_stream())
        outs = [yd, yt]
    else:
        x = torch.empty((5, K), dtype=torch.bfloat16, device=dev)
        y = torch.empty((5, N), device=dev)
        fn = q.cass_decode_draft if what == "draft" else q.cass_reconstruct
        call = lambda: fn(d, packed, x, y, None, torch.cuda.current_stream())
        outs = [y]
    _replay_matches(torch, call, [x], outs)
    assert q.qmv_check_status() == 0
