"""GPU parity of the MoE path (top-k routing over ternary SwiGLU experts) through the C ABI.

Checks: routing (experts and softmax weights) against the oracle; the gate/up
outputs per (token, expert) pair and the down projection + weighted combine
(fed the GPU's own h) within |err| <= 2e-3 * sum |w_hat x|; and the end-to-end
output within the bound those two give exactly: the down matvec's bound on the
GPU's own h, plus the down matrix applied to |h_gpu - h_exact|, plus the fp32
evaluation of silu(g) u and of the weighted combine.
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


class Experts:
    """E ternary SwiGLU experts packed as [gate; up] (2I x H) + down (H x I) records, fp32 masters kept on the GPU."""

    def __init__(self, q, torch, dev, E, H, I, seed, zero_cols=None, layout="record"):
        from quantized_gemv_unpack_gb300 import synth
        gen = synth.torch_generator(seed, dev)
        fmt = q.QMV_TERNARY2_LUT if layout == "lut" else q.QMV_TERNARY2
        self.gu_desc = q.qmv_pack_desc(fmt, 2 * I, H)
        self.dn_desc = q.qmv_pack_desc(fmt, H, I)
        self.down_off = self.gu_desc.total_bytes
        self.stride = self.down_off + self.dn_desc.total_bytes
        self.buf = torch.empty(E * self.stride, dtype=torch.uint8, device=dev)
        self.w_gu, self.w_dn = [], []
        for e in range(E):
            wgu = synth.student_t4_torch(gen, (2 * I, H), device=dev)
            wdn = synth.student_t4_torch(gen, (H, I), device=dev)
            if zero_cols is not None and len(zero_cols):
                # the outlier channels' weights are 0 in every even gate/up row
                wgu[0::2, torch.as_tensor(zero_cols, device=dev)] = 0.0
            rec = self.buf[e * self.stride:(e + 1) * self.stride]
            q.qmv_pack_ternary(self.gu_desc, wgu, rec[:self.down_off])
            q.qmv_pack_ternary(self.dn_desc, wdn, rec[self.down_off:])
            self.w_gu.append(wgu)
            self.w_dn.append(wdn)
        self.E, self.H, self.I = E, H, I

    def dequant_rows(self, which, e, rows):
        """Oracle-side dequantized rows (float64) of expert e's [gate; up] or down matrix."""
        from oracle import ternary
        w = (self.w_gu if which == "gu" else self.w_dn)[e]
        q_, _, s16 = ternary.quantize(w[rows].cpu().numpy())
        return ternary.dequant(q_, s16)


def _ws_views(q, ws, E, topk, M, I):
    """Views of the documented workspace layout (slots, pairs, g|u)."""
    import ctypes
    al = lambda v: (v + 255) // 256 * 256
    P, S = M * topk, min(E, M * topk)
    off_se = al(16)
    off_sf = al(off_se + 4 * S)
    off_sc = al(off_sf + 4 * S)
    off_pt = al(off_sc + 4 * S)
    off_pp = al(off_pt + 4 * P)
    off_gu = al(off_pp + 4 * P)
    h = ws.cpu().numpy()
    i32 = lambda o, n: h[o:o + 4 * n].view(np.int32)
    f32 = lambda o, n: h[o:o + 4 * n].view(np.float32)
    ns = int(i32(0, 1)[0])
    return dict(n_slots=ns, slot_expert=i32(off_se, S)[:ns], slot_first=i32(off_sf, S)[:ns],
                slot_count=i32(off_sc, S)[:ns], pair_token=i32(off_pt, P), pair_prob=f32(off_pp, P),
                gu=f32(off_gu, P * 2 * I).reshape(P, 2 * I))


def _run(q, torch, dev, ex, M, topk, seed, x=None):
    from quantized_gemv_unpack_gb300 import synth
    gen = synth.torch_generator(seed, dev)
    logits = synth.router_logits_torch(gen, M, ex.E, device=dev)
    if x is None:
        x = synth.activations_bf16_torch(gen, (M, ex.H), device=dev)
    y = torch.full((M, ex.H), float("nan"), device=dev)
    ws = torch.zeros(q.moe_workspace_size(ex.E, topk, M, ex.H, ex.I), dtype=torch.uint8, device=dev)
    q.moe_qmv_run(ex.gu_desc, ex.dn_desc, ex.buf, ex.stride, ex.down_off, ex.E, logits, topk, x, y, ws)
    assert q.qmv_check_status() == 0
    xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
    return logits.cpu().numpy(), xb, y.cpu().numpy(), _ws_views(q, ws, ex.E, topk, M, ex.I)


def _check_routing(logits, topk, W):
    from oracle import moe
    idx, p = moe.route(logits, topk)
    M = logits.shape[0]
    pairs = {}
    for s in range(W["n_slots"]):
        e = int(W["slot_expert"][s])
        for j in range(W["slot_first"][s], W["slot_first"][s] + W["slot_count"][s]):
            pairs[(int(W["pair_token"][j]), e)] = (j, float(W["pair_prob"][j]))
    assert len(pairs) == M * topk
    for t in range(M):
        for k in range(topk):
            j, pr = pairs[(t, int(idx[t, k]))]
            assert abs(pr - p[t, k]) <= 1e-6
    assert list(W["slot_expert"]) == sorted(set(int(v) for v in idx.ravel()))
    return idx, p, pairs


FP32_SLACK = 2e-6   # silu(g) * u and the combine in fp32: a few roundings of 2^-24 each


@pytest.mark.parametrize("layout", ["record", "lut"])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
@pytest.mark.parametrize("outliers", [None, "channels", "range"])
def test_moe_small_end_to_end(env, M, outliers, layout):
    q, torch, dev = env
    from oracle import moe
    from oracle.numerics import bf16_bits_to_f64
    from quantized_gemv_unpack_gb300 import synth
    E, H, I, topk = 16, 512, 256, 4
    xin, ch = None, None
    if outliers:
        xf, ch = synth.outlier_activations(synth.rng(60 + M), outliers, M, H)
        xin = torch.from_numpy(synth.to_bf16_bits(xf).view(np.int16)).to(dev).view(torch.bfloat16)
    ex = Experts(q, torch, dev, E, H, I, seed=30 + M, zero_cols=ch, layout=layout)
    logits, xb, y, W = _run(q, torch, dev, ex, M, topk, seed=M, x=xin)
    idx, p, pairs = _check_routing(logits, topk, W)
    x = bf16_bits_to_f64(xb)
    full = lambda which, e: ex.dequant_rows(which, e, torch.arange((2 * I) if which == "gu" else H, device=dev))
    cache = {}

    def weights(e):
        if e not in cache:
            gu_ = full("gu", e)
            cache[e] = (gu_[:I], gu_[I:], full("dn", e))
        return cache[e]

    yr, _, _, parts = moe.moe(x, logits, topk, weights)
    bound = np.zeros_like(yr)
    for (t, e), (pw, g, u, h, out) in parts.items():
        wg, wu, wd = weights(e)
        j, _ = pairs[(t, e)]
        # staged: g|u of this pair within the matvec bound
        Bg, Bu = np.abs(wg) @ np.abs(x[t]), np.abs(wu) @ np.abs(x[t])
        assert np.all(np.abs(W["gu"][j, :I] - g) <= RTOL * Bg)
        assert np.all(np.abs(W["gu"][j, I:] - u) <= RTOL * Bu)
        # the GPU's own h, and what its deviation from the exact h does through W_down
        gg = W["gu"][j, :I].astype(np.float64)
        ug = W["gu"][j, I:].astype(np.float64)
        hg = gg / (1.0 + np.exp(-gg)) * ug
        Bd = np.abs(wd) @ np.abs(hg)
        # plus the routing weight's own error (|p_gpu - p| <= 1e-6, checked above) times |out|
        bound[t] += pw * ((RTOL + FP32_SLACK) * Bd + np.abs(wd) @ np.abs(hg - h)) + 1e-6 * Bd
    assert np.all(np.abs(y - yr) <= bound + 1e-30), f"worst |err|/bound = {np.max(np.abs(y - yr) / np.maximum(bound, 1e-300)):.3f}"


@pytest.mark.parametrize("layout", ["record", "lut"])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_moe_full_size_staged(env, M, layout):
    """128 experts, hidden 4096, SwiGLU 2048, top-8: routing exact, g|u and down+combine on sampled rows,
    with the experts in the record layout (fp16-FMA expert kernels) or the byte-lookup layout
    (lookup kernel, one (token, expert) pair per task)."""
    q, torch, dev = env
    E, H, I, topk = 128, 4096, 2048, 8
    ex = Experts(q, torch, dev, E, H, I, seed=3, layout=layout)
    logits, xb, y, W = _run(q, torch, dev, ex, M, topk, seed=100 + M)
    idx, p, pairs = _check_routing(logits, topk, W)
    from oracle.numerics import bf16_bits_to_f64
    x = bf16_bits_to_f64(xb)
    rng = np.random.default_rng(M)
    gu_rows = np.unique(np.concatenate(([0, I - 1, I, 2 * I - 1], rng.choice(2 * I, 12, replace=False))))
    dn_rows = np.unique(np.concatenate(([0, H - 1], rng.choice(H, 14, replace=False))))
    yr = np.zeros((M, len(dn_rows)))
    yb = np.zeros((M, len(dn_rows)))
    for (t, e), (j, pw) in pairs.items():
        wg = ex.dequant_rows("gu", e, torch.from_numpy(gu_rows).to(dev))
        ref = wg @ x[t]
        B = np.abs(wg) @ np.abs(x[t])
        assert np.all(np.abs(W["gu"][j, gu_rows] - ref) <= RTOL * B)
        g = W["gu"][j, :I].astype(np.float64)
        u = W["gu"][j, I:].astype(np.float64)
        h = g / (1.0 + np.exp(-g)) * u                     # the GPU's own g and u
        wd = ex.dequant_rows("dn", e, torch.from_numpy(dn_rows).to(dev))
        yr[t] += pw * (wd @ h)
        yb[t] += pw * (np.abs(wd) @ np.abs(h))
    assert np.all(np.abs(y[:, dn_rows] - yr) <= (RTOL + FP32_SLACK) * yb)


def test_moe_rejects_bad_arguments(env):
    q, torch, dev = env
    ex = Experts(q, torch, dev, 4, 256, 128, seed=1)
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((1, 256), device=dev)
    logits = torch.zeros((1, 4), device=dev)
    ws = torch.zeros(q.moe_workspace_size(4, 2, 1, 256, 128), dtype=torch.uint8, device=dev)
    with pytest.raises(q.QmvError):
        q.moe_qmv_run(ex.gu_desc, ex.dn_desc, ex.buf, ex.stride, ex.down_off, 4, logits, 5, x, y, ws)   # topk > E
    with pytest.raises(q.QmvError):
        q.moe_qmv_run(ex.gu_desc, ex.dn_desc, ex.buf, ex.stride, ex.down_off, 4, logits, 2, x, y, ws[:64])
    with pytest.raises(q.QmvError):
        q.moe_qmv_run(ex.dn_desc, ex.gu_desc, ex.buf, ex.stride, ex.down_off, 4, logits, 2, x, y, ws)


def _edge_logits(kind, M, E, seed):
    """Router logits with the hard cases of the selection: many equal logits (the lower
    expert first), signed zeros (equal), NaN entries (ranked as -inf; every token keeps at
    least k finite logits, so none is selected)."""
    g = np.random.default_rng(seed)
    if kind == "random":
        return g.standard_normal((M, E)).astype(np.float32)
    if kind == "ties":
        return g.choice(np.array([-1.0, 0.0, 0.5, 1.0], np.float32), size=(M, E))
    if kind == "zeros":
        z = g.choice(np.array([0.0, -0.0, 0.25], np.float32), size=(M, E))
        return z.astype(np.float32)
    if kind == "nan":
        lg = g.standard_normal((M, E)).astype(np.float32)
        for t in range(M):
            lg[t, g.choice(E, size=E // 3, replace=False)] = np.nan
        return lg
    raise ValueError(kind)


@pytest.mark.parametrize("layout", ["record", "lut"])
@pytest.mark.parametrize("E,topk,M", [(1, 1, 1), (7, 3, 2), (40, 8, 8), (129, 2, 3), (200, 8, 5), (256, 8, 8)])
@pytest.mark.parametrize("kind", ["random", "ties", "zeros", "nan"])
def test_routing_edge_cases(env, layout, E, topk, M, kind):
    # the routing every expert CTA computes, read back from the workspace, against the oracle's
    # top-k (larger logit first, equal logits lower expert first) and softmax
    q, torch, dev = env
    H = I = 128
    ex = _small_experts(q, torch, dev, E, H, I, layout)
    lg = _edge_logits(kind, M, E, seed=E * 100 + M)
    if kind == "nan":
        assert all(np.isfinite(lg[t]).sum() >= topk for t in range(M))
    logits = torch.from_numpy(lg).to(dev)
    x = torch.from_numpy(np.zeros((M, H), np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((M, H), device=dev)
    ws = torch.zeros(q.moe_workspace_size(E, topk, M, H, I), dtype=torch.uint8, device=dev)
    q.moe_qmv_run(ex.gu_desc, ex.dn_desc, ex.buf, ex.stride, ex.down_off, E, logits, topk, x, y, ws)
    assert q.qmv_check_status() == 0
    lg_oracle = np.where(np.isnan(lg), -np.inf, lg).astype(np.float32)
    _check_routing(lg_oracle, topk, _ws_views(q, ws, E, topk, M, I))
    assert np.all(y.cpu().numpy() == 0.0)   # x = 0: every expert output is 0


_SMALL = {}


def _small_experts(q, torch, dev, E, H, I, layout):
    key = (E, H, I, layout)
    if key not in _SMALL:
        _SMALL.clear()
        _SMALL[key] = Experts(q, torch, dev, E, H, I, seed=E, layout=layout)
    return _SMALL[key]
