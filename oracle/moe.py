"""MoE decode with top-k routing over ternary SwiGLU experts. TEST INFRASTRUCTURE ONLY.

"Nemotron 3.5 Bolt" (expert top-K routing section) activates a fixed top-K of
the experts per token, so a decode step reads only the active experts'
weights. Per token t with router logits l_t over E experts:

* the top-k experts by logit (equal logits: lower expert index first);
* p_{t,e} = softmax over the k selected logits (float64);
* expert e: g = W_gate x, u = W_up x, h = silu(g) * u = g * sigmoid(g) * u,
  out = W_down h;
* y_t = sum over the selected e of p_{t,e} * out_{t,e}.

Expert weights come in as dequantized float64 matrices from ``oracle.ternary``.
"""
from __future__ import annotations

import numpy as np


def route(logits: np.ndarray, topk: int):
    """logits float32 [M][E] -> (experts int [M][topk], p float64 [M][topk])."""
    logits = np.asarray(logits, dtype=np.float32)
    M, E = logits.shape
    idx = np.broadcast_to(np.arange(E), (M, E))
    order = np.lexsort((idx, -logits.astype(np.float64)), axis=1)[:, :topk]
    sel = np.take_along_axis(logits.astype(np.float64), order, axis=1)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    return order, p


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def expert_forward(w_gate, w_up, w_down, x: np.ndarray):
    """x float64 [T][H] -> (g, u, h, out) for one expert, all float64."""
    g = x @ w_gate.T
    u = x @ w_up.T
    h = silu(g) * u
    return g, u, h, h @ w_down.T


def moe(x: np.ndarray, logits: np.ndarray, topk: int, expert_weights):
    """y float64 [M][H]; expert_weights(e) -> (w_gate, w_up, w_down) float64.

    Also returns per-token, per-slot intermediate values for staged checks:
    dict (t, e) -> (p, g, u, h, out).
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    M, H = x.shape
    experts, p = route(logits, topk)
    y = np.zeros((M, H), dtype=np.float64)
    parts = {}
    for e in sorted(set(int(v) for v in experts.ravel())):
        toks = [t for t in range(M) if e in experts[t]]
        wg, wu, wd = expert_weights(e)
        g, u, h, out = expert_forward(wg, wu, wd, x[toks])
        for i, t in enumerate(toks):
            slot = int(np.where(experts[t] == e)[0][0])
            y[t] += p[t, slot] * out[i]
            parts[(t, e)] = (p[t, slot], g[i], u[i], h[i], out[i])
    return y, experts, p, parts
