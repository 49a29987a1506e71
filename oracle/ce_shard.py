"""fp64 oracle of the vocabulary-sharded cross-entropy (test infrastructure).

What it computes ("Add Megatron-LM cross-entropy integration", Summary: the
vocab-parallel CE of a tensor-parallel group; "Add opt-in Liger vocab-parallel
cross entropy through ops/loss", What does this PR do: the global argmax and
the merge of per-shard statistics over the group): each rank holds the columns
[vocab_start, vocab_start + V_local) of every row of the logits.  Per row and
shard it forms

    x_max, argmax   the shard's largest raw logit and its smallest global column
    lse             log sum_j exp(z_j) over the shard's columns
    sum_z           sum_j z_j over the shard's columns
    z_y             z at the label column if the shard holds it, else 0

(z = T tanh(x/T) with softcap T > 0, else z = x); the statistics of the whole
vocabulary are the merge of the shards' (largest x_max, smallest index on
ties; log-add-exp of lse; sums of sum_z and z_y), from which every rank forms
the row's loss and the gradient of its own columns exactly as the unsharded
cross-entropy does.  Plain numpy in fp64; the gradient columns come from the
CE oracle's grad_columns.  Only the tests use this module.
"""
from __future__ import annotations

import numpy as np
from scipy.special import logsumexp

from . import ce


def _z(x: np.ndarray, softcap: float) -> np.ndarray:
    return softcap * np.tanh(x / softcap) if softcap > 0 else x


def shard_stats(x: np.ndarray, vocab_start: int, labels: np.ndarray, softcap: float = 0.0) -> dict:
    """x: fp64 [n, V_local] raw logits of the shard.  Statistics per row."""
    x = np.asarray(x, np.float64)
    n, vl = x.shape
    labels = np.asarray(labels, np.int64)
    z = _z(x, softcap)
    rows = np.arange(n)
    local = labels - vocab_start
    mine = (local >= 0) & (local < vl)
    z_y = np.zeros(n)
    z_y[mine] = z[rows[mine], local[mine]]
    return dict(x_max=x.max(axis=1), argmax=vocab_start + x.argmax(axis=1),  # first occurrence
                lse=logsumexp(z, axis=1), sum_z=z.sum(axis=1), z_y=z_y)


def merge_stats(parts: list[dict]) -> dict:
    """Merge shard statistics in the given order."""
    out = {k: np.array(v, copy=True) for k, v in parts[0].items()}
    for p in parts[1:]:
        take = (p["x_max"] > out["x_max"]) | ((p["x_max"] == out["x_max"]) &
                                              (p["argmax"] < out["argmax"]))
        out["x_max"] = np.where(take, p["x_max"], out["x_max"])
        out["argmax"] = np.where(take, p["argmax"], out["argmax"])
        out["lse"] = np.logaddexp(out["lse"], p["lse"])
        out["sum_z"] = out["sum_z"] + p["sum_z"]
        out["z_y"] = out["z_y"] + p["z_y"]
    return out


def row_loss(stats: dict, labels: np.ndarray, V: int, *, ignore_index: int = -100,
             label_smoothing: float = 0.0) -> np.ndarray:
    """Per-row loss from the whole vocabulary's statistics (NaN for a bad label)."""
    labels = np.asarray(labels, np.int64)
    eps = label_smoothing
    valid = (labels != ignore_index) & (labels >= 0) & (labels < V)
    loss = np.where(valid, stats["lse"] - (1 - eps) * stats["z_y"] - (eps / V) * stats["sum_z"],
                    0.0)
    return np.where(~valid & (labels != ignore_index), np.nan, loss)


def shard_grad(x: np.ndarray, vocab_start: int, V: int, labels: np.ndarray, lse: np.ndarray,
               row_scale: np.ndarray, *, ignore_index: int = -100, label_smoothing: float = 0.0,
               softcap: float = 0.0) -> np.ndarray:
    """Gradient of the shard's columns given the rows' global lse and scale."""
    x = np.asarray(x, np.float64)
    cols = vocab_start + np.arange(x.shape[1])
    return ce.grad_columns(x, cols, V, labels, lse, row_scale, ignore_index=ignore_index,
                           label_smoothing=label_smoothing, softcap=softcap)


def sharded_fwd_bwd(x: np.ndarray, bounds: list[int], labels: np.ndarray, *,
                    ignore_index: int = -100, label_smoothing: float = 0.0, softcap: float = 0.0,
                    reduction: str = "mean", grad_scale: float = 1.0) -> dict:
    """The whole protocol on fp64 logits [n, V] cut at column `bounds` (0 < b < V):
    statistics per shard, merge, loss and per-shard gradients (joined)."""
    x = np.asarray(x, np.float64)
    n, V = x.shape
    labels = np.asarray(labels, np.int64)
    edges = [0] + list(bounds) + [V]
    parts = [shard_stats(x[:, a:b], a, labels, softcap) for a, b in zip(edges[:-1], edges[1:])]
    g = merge_stats(parts)
    loss = row_loss(g, labels, V, ignore_index=ignore_index, label_smoothing=label_smoothing)
    n_valid, _ = ce.count(labels, V, ignore_index)
    s = ce.scale(reduction, grad_scale, n_valid)
    valid = (labels != ignore_index) & (labels >= 0) & (labels < V)
    sc = np.where(valid, s, 0.0)
    grad = np.concatenate([shard_grad(x[:, a:b], a, V, labels, g["lse"], sc,
                                      ignore_index=ignore_index, label_smoothing=label_smoothing,
                                      softcap=softcap)
                           for a, b in zip(edges[:-1], edges[1:])], axis=1)
    red, acc, n_correct = ce.reduce(loss, g["argmax"], labels, V, ignore_index, reduction)
    return dict(loss=loss, argmax=g["argmax"], grad=grad, reduced_loss=red, accuracy=acc,
                n_valid=n_valid, n_correct=n_correct, stats=g)
