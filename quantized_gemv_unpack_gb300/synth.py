"""Seeded synthetic inputs shared by the CUDA path, the tests and the benchmark.

This module only draws random numbers. It quantizes nothing, packs nothing and
computes no part of the method; both the oracle-side checks and the CUDA side
receive the arrays it returns as plain inputs.

Distributions follow the workloads the pages measure on:

* weights: Student-t with 4 degrees of freedom, rescaled to a standard
  deviation of 0.02 (heavy-tailed, peaked weights as described in the
  "Ternary Bonsai 2" page, section 1.2). A t(4) variate is drawn as
  Z / sqrt(V / 4) with Z ~ N(0, 1) and V ~ chi-square(4) = -2 (ln U1 + ln U2);
  t(4) has variance 4 / (4 - 2) = 2, so the draw is multiplied by 0.02 / sqrt(2).
* activations: N(0, 1) rounded to bfloat16 (round to nearest even).
* Cassandra calibration rows: N(0, 1) with 1 % of the channels (a seeded
  permutation, floor(0.01 K) channels) multiplied by 20 before the bf16
  rounding, so that the Wanda norm sees outlier channels ("Cassandra" page,
  section 3.2).
* MoE router logits: N(0, 1) in float32.
* outlier activations (parity edge cases): LLM activations carry a few
  channels far larger than the rest (the "Cassandra" page's calibration scales
  1 % of the channels by 20); `outlier_case` makes 1 % of the channels 1000x
  the rest, or one channel 2^24x, with zero weights on those columns in every
  even row, or spreads magnitudes log-uniformly over a 2^24 range.

Two back ends produce the same distributions from different streams: NumPy
(PCG64) on the host for sizes the oracle can handle, and torch (Philox) on the
GPU for the multi-gigabyte stack and expert sets. A given test or benchmark
uses one back end for both sides.
"""
from __future__ import annotations

import math

import numpy as np

T4_STD = math.sqrt(2.0)


# ----------------------------------------------------------------------------- numpy

def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def student_t4(g: np.random.Generator, shape, std: float = 0.02) -> np.ndarray:
    """float32 Student-t(4) samples with the given standard deviation."""
    z = g.standard_normal(shape, dtype=np.float64)
    u1 = 1.0 - g.random(shape, dtype=np.float64)  # (0, 1]
    u2 = 1.0 - g.random(shape, dtype=np.float64)
    v = -2.0 * (np.log(u1) + np.log(u2))
    t = z / np.sqrt(v / 4.0)
    return (t * (std / T4_STD)).astype(np.float32)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even) and return the raw uint16 bits.

    NaN inputs never occur in the generated data, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations_bf16(g: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) activations as raw bfloat16 bits (uint16)."""
    return to_bf16_bits(g.standard_normal(shape, dtype=np.float32))


def calibration_bf16(g: np.random.Generator, rows: int, K: int,
                     outlier_frac: float = 0.01, outlier_gain: float = 20.0):
    """Calibration activations [rows][K] as bf16 bits, plus the outlier channels."""
    x = g.standard_normal((rows, K), dtype=np.float32)
    n_out = int(math.floor(outlier_frac * K))
    chans = np.sort(g.permutation(K)[:n_out])
    x[:, chans] *= np.float32(outlier_gain)
    return to_bf16_bits(x), chans


def router_logits(g: np.random.Generator, M: int, E: int) -> np.ndarray:
    return g.standard_normal((M, E), dtype=np.float32)


OUTLIER_KINDS = ("channels", "huge", "range")


def outlier_activations(g: np.random.Generator, kind: str, M: int, K: int):
    """float32 activations [M][K] with an extreme range inside each row, and the columns
    whose weights the caller should zero in some rows (empty for "range").

    "channels": floor(1 % of K) channels (at least one, a seeded permutation) 1000x an
    N(0, 1) draw; "huge": one channel at +-2^24; "range": sign of an N(0, 1) draw times
    2^u, u uniform on [-12, 12]."""
    x = g.standard_normal((M, K)).astype(np.float32)
    if kind == "channels":
        ch = np.sort(g.permutation(K)[: max(1, K // 100)])
        x[:, ch] *= np.float32(1000.0)
    elif kind == "huge":
        ch = np.array([int(g.integers(0, K))])
        x[:, ch] = np.float32(2.0 ** 24) * np.where(g.random((M, 1)) < 0.5, -1, 1).astype(np.float32)
    elif kind == "range":
        ch = np.zeros(0, dtype=np.int64)
        x = (np.sign(x) * np.exp2(g.uniform(-12, 12, size=(M, K)))).astype(np.float32)
    else:
        raise ValueError(kind)
    return x, ch


def outlier_case(kind: str, N: int, K: int, M: int, seed: int):
    """Student-t weights [N][K] (float32) whose outlier columns are 0 in every even row,
    and `outlier_activations` of that kind as bf16 bits [M][K]."""
    g = rng(seed)
    w = student_t4(g, (N, K))
    x, ch = outlier_activations(g, kind, M, K)
    if len(ch):
        w[0::2, :][:, ch] = 0.0
    return w, to_bf16_bits(x)


# ----------------------------------------------------------------------------- torch

def torch_generator(seed: int, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def student_t4_torch(gen, shape, std: float = 0.02, device="cuda", out=None):
    """float32 Student-t(4) samples drawn on `device` with a torch generator."""
    import torch
    z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    u = torch.rand((2,) + tuple(shape), generator=gen, device=device, dtype=torch.float32)
    u = 1.0 - u  # (0, 1]
    v = -2.0 * (torch.log(u[0]) + torch.log(u[1]))
    del u
    t = z / torch.sqrt(v * 0.25)
    del z, v
    t.mul_(std / T4_STD)
    if out is not None:
        out.copy_(t)
        return out
    return t


def activations_bf16_torch(gen, shape, device="cuda"):
    import torch
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def router_logits_torch(gen, M: int, E: int, device="cuda"):
    import torch
    return torch.randn((M, E), generator=gen, device=device, dtype=torch.float32)


# ----------------------------------------------------------------------------- shapes

def gqa_layer_shapes(hidden: int, n_q: int, n_kv: int, head_dim: int, inter: int):
    """(name, N, K) of the seven linear maps of one GQA + SwiGLU block."""
    q = n_q * head_dim
    kv = n_kv * head_dim
    return [("q", q, hidden), ("k", kv, hidden), ("v", kv, hidden), ("o", hidden, q),
            ("gate", inter, hidden), ("up", inter, hidden), ("down", hidden, inter)]
