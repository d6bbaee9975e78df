"""moe_qmv_run_static: the MoE decode for callers that cannot allocate device memory.

Such callers (a plugin whose host application owns every device allocation, or
a loop that must not pay for cudaMalloc) pass no workspace; the library uses a
fixed scratch array in its own device memory instead. This test calls the
entry point through the C ABI twice in a row and checks each output against
the workspace entry point, moe_qmv_run, within the tolerance the MoE tests use
(|dy| <= 2e-3 * sum_e p_e sum_i |w_down h|, with h from the GPU's own gate/up
outputs). It also checks that a call needing more scratch than the array holds
is refused before anything runs. It lives in a file of its own so that pytest
collects it last.
"""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]

RTOL = 2e-3


def test_static_scratch_matches_workspace_entry_point():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_gemv_unpack_gb300 as q
    from oracle import ternary
    from quantized_gemv_unpack_gb300 import synth

    dev = torch.device("cuda:0")
    E, H, I, topk, M = 16, 512, 256, 4, 3
    gen = synth.torch_generator(77, dev)
    gu_desc = q.qmv_pack_desc(q.QMV_TERNARY2, 2 * I, H)
    dn_desc = q.qmv_pack_desc(q.QMV_TERNARY2, H, I)
    down_off = gu_desc.total_bytes
    stride = down_off + dn_desc.total_bytes
    experts = torch.empty(E * stride, dtype=torch.uint8, device=dev)
    w_dn = []
    for e in range(E):
        rec = experts[e * stride:(e + 1) * stride]
        q.qmv_pack_ternary(gu_desc, synth.student_t4_torch(gen, (2 * I, H), device=dev), rec[:down_off])
        wd = synth.student_t4_torch(gen, (H, I), device=dev)
        q.qmv_pack_ternary(dn_desc, wd, rec[down_off:])
        w_dn.append(wd.cpu().numpy())
    logits = synth.router_logits_torch(gen, M, E, device=dev)
    x = synth.activations_bf16_torch(gen, (M, H), device=dev)

    # reference: the workspace entry point, keeping its workspace to read g and u
    ws = torch.zeros(q.moe_workspace_size(E, topk, M, H, I), dtype=torch.uint8, device=dev)
    y_ws = torch.empty((M, H), device=dev)
    q.moe_qmv_run(gu_desc, dn_desc, experts, stride, down_off, E, logits, topk, x, y_ws, ws)
    assert q.qmv_check_status() == 0

    # the bound: sum over each token's experts of p * sum_i |w_down[row, i] * h_i|, h from the GPU's g and u
    al = lambda v: (v + 255) // 256 * 256
    P, S = M * topk, min(E, M * topk)
    off_pt = al(al(al(al(16) + 4 * S) + 4 * S) + 4 * S)
    off_pp = al(off_pt + 4 * P)
    off_gu = al(off_pp + 4 * P)
    h = ws.cpu().numpy()
    ns = int(h[:4].view(np.int32)[0])
    slot_expert = h[al(16):al(16) + 4 * S].view(np.int32)[:ns]
    slot_first = h[al(al(16) + 4 * S):al(al(16) + 4 * S) + 4 * S].view(np.int32)[:ns]
    slot_count = h[al(al(al(16) + 4 * S) + 4 * S):al(al(al(16) + 4 * S) + 4 * S) + 4 * S].view(np.int32)[:ns]
    pair_token = h[off_pt:off_pt + 4 * P].view(np.int32)
    pair_prob = h[off_pp:off_pp + 4 * P].view(np.float32)
    gu = h[off_gu:off_gu + 4 * P * 2 * I].view(np.float32).reshape(P, 2 * I).astype(np.float64)
    bound = np.zeros((M, H))
    for s in range(ns):
        e = int(slot_expert[s])
        qq, _, s16 = ternary.quantize(w_dn[e])
        wd_hat = np.abs(ternary.dequant(qq, s16))
        for j in range(slot_first[s], slot_first[s] + slot_count[s]):
            g, u = gu[j, :I], gu[j, I:]
            hj = g / (1.0 + np.exp(-g)) * u
            bound[pair_token[j]] += pair_prob[j] * (wd_hat @ np.abs(hj))
    assert np.all(bound > 0)

    ref = y_ws.cpu().numpy()
    for _ in range(2):  # two calls in a row: the shared scratch keeps the previous call's contents
        y = torch.full((M, H), float("nan"), device=dev)
        q.moe_qmv_run_static(gu_desc, dn_desc, experts, stride, down_off, E, logits, topk, x, y)
        assert q.qmv_check_status() == 0
        assert np.all(np.abs(y.cpu().numpy() - ref) <= RTOL * bound)

    # a call that needs more scratch than the array holds is refused before any launch
    big_gu = q.qmv_pack_desc(q.QMV_TERNARY2, 2 * 32768, 128)
    big_dn = q.qmv_pack_desc(q.QMV_TERNARY2, 128, 32768)
    big_stride = big_gu.total_bytes + big_dn.total_bytes
    assert q.moe_workspace_size(8, 8, 8, 128, 32768) > q.QMV_MOE_STATIC_SCRATCH_BYTES
    small = torch.zeros(1024, dtype=torch.uint8, device=dev)
    xs = torch.zeros((8, 128), dtype=torch.bfloat16, device=dev)
    ys = torch.zeros((8, 128), device=dev)
    lg = torch.zeros((8, 8), device=dev)
    with pytest.raises(q.QmvError) as err:
        q.moe_qmv_run_static(big_gu, big_dn, small, big_stride, big_gu.total_bytes, 8, lg, 8, xs, ys)
    assert err.value.status == q.QMV_ERR_ARG and "static scratch" in str(err.value)
