"""fp64 oracle for the fused linear cross-entropy (test infrastructure).

What it computes ("Add Liger Kernel support for Muse Glimmer", Summary and
Details: Softcap): the logits are the plain product S = h' W^T of the hidden
states (already multiplied by the logit multiplier m) and the lm_head weight,
the cross-entropy of the CE oracle is applied to S, and the gradients follow
from G = dLoss/dS (the CE oracle's gradient):

    grad_hidden = G W        grad_weight = G^T h'

Matrix products are fp64 library matmuls (numpy); everything else is the CE
oracle (``oracle/ce_oracle.c``).  Only the tests, the smoke check and the
benchmark's CPU legs use this module.

Two ways in:
* :func:`flce_fwd_bwd` -- everything at once (small shapes);
* :func:`sampled` -- any size: the weight is streamed in vocabulary blocks
  (the per-row log-sum-exp is the log of the sum of the blocks' exp-sums,
  ``np.logaddexp``), losses and argmaxes come for every row, the hidden
  gradient for sampled rows and the weight gradient for sampled vocabulary
  rows.
"""
from __future__ import annotations

import numpy as np
from scipy.special import logsumexp

from . import ce


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64, exactly."""
    return (np.ascontiguousarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def flce_fwd_bwd(h: np.ndarray, W: np.ndarray, labels: np.ndarray, *, ignore_index: int = -100,
                 label_smoothing: float = 0.0, softcap: float = 0.0, reduction: str = "mean",
                 grad_scale: float = 1.0, want_grad: bool = True) -> dict:
    """h: fp64 [N, H] (h' = m h); W: fp64 [V, H].  Returns the CE oracle's dict
    for the logits S = h W^T plus grad_hidden [N, H] and grad_weight [V, H]."""
    V = W.shape[0]
    S = h @ W.T
    r = ce.ce_fwd_bwd(S, "f64", V, labels, ignore_index=ignore_index,
                      label_smoothing=label_smoothing, softcap=softcap, reduction=reduction,
                      grad_scale=grad_scale, want_grad=want_grad)
    if want_grad:
        r["grad_hidden"] = r["grad"] @ W
        r["grad_weight"] = r["grad"].T @ h
    return r


def _z(S: np.ndarray, softcap: float) -> np.ndarray:
    return softcap * np.tanh(S / softcap) if softcap > 0 else S


def row_stats(h: np.ndarray, W_bits: np.ndarray, labels: np.ndarray, *, softcap: float = 0.0,
              block: int = 8192) -> dict:
    """Per row over the whole vocabulary, W (bf16 bits [V, H]) streamed in
    blocks of `block` rows: lse of z, first argmax of S, z at the label, sum z,
    and the two largest logits S (``top``, ``second``: the largest two entries
    of the row counted with multiplicity, so a duplicated maximum gives
    second = top).  top - second is how close a row is to an argmax tie."""
    N = h.shape[0]
    V = W_bits.shape[0]
    lse = np.full(N, -np.inf)
    best = np.full(N, -np.inf)
    second = np.full(N, -np.inf)
    amax = np.zeros(N, np.int64)
    zy = np.zeros(N)
    sumz = np.zeros(N)
    rows = np.arange(N)
    for v0 in range(0, V, block):
        v1 = min(V, v0 + block)
        S = h @ widen_bf16(W_bits[v0:v1]).T
        z = _z(S, softcap)
        lse = np.logaddexp(lse, logsumexp(z, axis=1))
        bm = S.max(axis=1)
        bi = S.argmax(axis=1)  # first occurrence in the block
        # the block's second largest (with multiplicity), merged with the running pair
        b2 = np.partition(S, -2, axis=1)[:, -2] if S.shape[1] >= 2 else np.full(N, -np.inf)
        second = np.maximum(np.minimum(best, bm), np.maximum(second, b2))
        upd = bm > best        # strictly greater: earlier blocks keep ties
        best = np.where(upd, bm, best)
        amax = np.where(upd, v0 + bi, amax)
        sumz += z.sum(axis=1)
        inb = (labels >= v0) & (labels < v1)
        zy[inb] = z[rows[inb], labels[inb] - v0]
    return dict(lse=lse, argmax=amax, zy=zy, sumz=sumz, top=best, second=second)


def sampled(h_bits: np.ndarray, W_bits: np.ndarray, labels: np.ndarray, rows, cols, *,
            ignore_index: int = -100, label_smoothing: float = 0.0, softcap: float = 0.0,
            reduction: str = "mean", grad_scale: float = 1.0, block: int = 8192) -> dict:
    """Loss, argmax, the two largest logits and reduced values of every row;
    grad_hidden of `rows`; grad_weight of vocabulary rows `cols`.  h_bits
    [N, H], W_bits [V, H]: bf16 bits."""
    h = widen_bf16(h_bits)
    V = W_bits.shape[0]
    labels = np.asarray(labels, np.int64)
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    n_valid, n_bad = ce.count(labels, V, ignore_index)
    s = ce.scale(reduction, grad_scale, n_valid)
    st = row_stats(h, W_bits, labels, softcap=softcap, block=block)
    eps = label_smoothing
    valid = (labels != ignore_index) & (labels >= 0) & (labels < V)
    ignored = labels == ignore_index
    loss = np.where(valid, st["lse"] - (1 - eps) * st["zy"] - (eps / V) * st["sumz"], 0.0)
    loss = np.where(~valid & ~ignored, np.nan, loss)
    red, acc, n_correct = ce.reduce(loss, st["argmax"], labels, V, ignore_index, reduction)
    # hidden gradient of the sampled rows: their full logits through the CE oracle
    out = dict(loss=loss, argmax=st["argmax"], lse=st["lse"], reduced_loss=red, accuracy=acc,
               n_valid=n_valid, n_correct=n_correct, n_bad=n_bad, row_scale=s, top=st["top"],
               second=st["second"])
    if rows.size:
        hR = h[rows]
        SR = np.concatenate([hR @ widen_bf16(W_bits[v0:v0 + block]).T
                             for v0 in range(0, V, block)], axis=1)
        _, _, GR = ce.rows(SR, "f64", V, labels[rows], ignore_index=ignore_index,
                           label_smoothing=eps, softcap=softcap, row_scale=s)
        gh = np.zeros((rows.size, h.shape[1]))
        for v0 in range(0, V, block):
            gh += GR[:, v0:v0 + block] @ widen_bf16(W_bits[v0:v0 + block])
        out["grad_hidden_rows"] = gh
    # weight gradient of the sampled vocabulary rows, from every row's lse
    if cols.size:
        Wc = widen_bf16(W_bits[cols])
        SC = h @ Wc.T
        GC = ce.grad_columns(SC, cols, V, labels, st["lse"], np.where(valid, s, 0.0),
                             ignore_index=ignore_index, label_smoothing=eps, softcap=softcap)
        out["grad_weight_cols"] = GC.T @ h
    return out
