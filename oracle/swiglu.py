"""fp64 oracle of the fused gate-up SwiGLU (test infrastructure).

What it computes ("[Megatron] Add SwiGLU integration", Summary and Background):
the fused first linear layer of a Megatron MLP produces one [tokens, 2n]
tensor with the gate in columns [0, n) and the up projection in [n, 2n); the
activation reads both halves of each row in place (row stride 2n) and writes

    y = silu(gate) * up,    silu(a) = a sigma(a),  sigma(a) = 1 / (1 + exp(-a))

(row stride n).  Its backward, given dy [tokens, n]:

    d_up   = dy * silu(gate)
    d_gate = dy * up * silu'(gate),  silu'(a) = sigma(a) (1 + a (1 - sigma(a)))

written to a [tokens, 2n] gradient in the same layout.  Plain numpy, fp64;
only the tests and the benchmark's CPU legs use this module.
"""
from __future__ import annotations

import numpy as np


def sigmoid(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, np.float64)
    out = np.empty_like(a)
    pos = a >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-a[pos]))
    e = np.exp(a[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def forward(x: np.ndarray, n: int) -> np.ndarray:
    """x: fp64 [T, 2n] (gate | up) -> y fp64 [T, n]."""
    x = np.asarray(x, np.float64)
    a, b = x[:, :n], x[:, n:2 * n]
    return a * sigmoid(a) * b


def backward(x: np.ndarray, dy: np.ndarray, n: int) -> np.ndarray:
    """x: fp64 [T, 2n], dy: fp64 [T, n] -> dx fp64 [T, 2n] (d_gate | d_up)."""
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    a, b = x[:, :n], x[:, n:2 * n]
    s = sigmoid(a)
    d_gate = dy * b * s * (1.0 + a * (1.0 - s))
    d_up = dy * a * s
    return np.concatenate([d_gate, d_up], axis=1)


def backward_terms(x: np.ndarray, dy: np.ndarray, n: int) -> np.ndarray:
    """Sum of the magnitudes of the products that make up each d_gate / d_up
    element (|dy b sigma| + |dy b a sigma (1 - sigma)| and |dy a sigma|): the
    scale of the rounding error of any fp32 evaluation."""
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    a, b = x[:, :n], x[:, n:2 * n]
    s = sigmoid(a)
    t_gate = np.abs(dy * b * s) + np.abs(dy * b * a * s * (1.0 - s))
    t_up = np.abs(dy * a * s)
    return np.concatenate([t_gate, t_up], axis=1)
