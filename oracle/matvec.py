"""float64 matvec y = W_hat x and the per-row error-bound term. TEST INFRASTRUCTURE ONLY.

The decode step every page turns on reads each weight once per token and forms
y = W x ("Nemotron 3.5 Bolt", why-only-weights section: weight-bandwidth-bound
low-batch decode). With M activation rows x[m] (1 token plus speculative
drafts), y[m][n] = sum_k w_hat[n][k] * x[m][k].

The comparison bound for a GPU result is |y - y_ref| <= rtol * B with
B[m][n] = sum_k |w_hat[n][k] * x[m][k]|.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_bits_to_f64


def matvec(w_hat: np.ndarray, x: np.ndarray):
    """w_hat float64 [N][K], x float64 [M][K] -> (y [M][N], B [M][N])."""
    w_hat = np.asarray(w_hat, dtype=np.float64)
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    y = x @ w_hat.T
    B = np.abs(x) @ np.abs(w_hat).T
    return y, B


def matvec_bf16x(w_hat: np.ndarray, x_bf16_bits: np.ndarray):
    return matvec(w_hat, bf16_bits_to_f64(x_bf16_bits))


def rows(w_hat_rows: np.ndarray, x: np.ndarray):
    """The same for a subset of rows (sampled checks at full size)."""
    return matvec(w_hat_rows, x)
