"""fp64 oracle for the cross-entropy forward + backward (test infrastructure).

Thin ctypes wrapper over ``ce_oracle.c``; the arithmetic lives there and is
documented there.  The shared library is compiled with gcc on first use (or
by ``__graft_entry__.build()``) next to the source.

Sources: "Add Megatron-LM cross-entropy integration" (Summary: ignore_index,
label_smoothing, online softmax with the gradient over the logits); "Add
opt-in Liger vocab-parallel cross entropy through ops/loss" (What does this
PR do: fp32 per-token loss, gradient dtype, smallest-index argmax); "Add Liger
Kernel support for Muse Glimmer" (Summary, Details: token accuracy, softcap).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ce_oracle.c")
_LIB = os.path.join(_HERE, "libce_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "bf16": 1, "f64": 2}
REDUCTIONS = {"none": 0, "mean": 1, "sum": 2}  # "none": per-token losses, gradient not averaged


def build(force: bool = False) -> str:
    """Compile ce_oracle.c into libce_oracle.so (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_GNU_SOURCE", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_ce_rows.argtypes = [vp, i32, i64, i64, i64, vp, i64, dbl, dbl, dbl, vp, vp,
                                           vp, i32]
            lib.oracle_ce_rows.restype = i32
            lib.oracle_ce_count.argtypes = [vp, i64, i64, i64, vp, vp]
            lib.oracle_ce_count.restype = None
            lib.oracle_ce_scale.argtypes = [i32, dbl, i64]
            lib.oracle_ce_scale.restype = dbl
            lib.oracle_ce_reduce.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, vp, vp]
            lib.oracle_ce_reduce.restype = None
            lib.oracle_round_bf16.argtypes = [vp, vp, i64]
            lib.oracle_round_bf16.restype = None
            lib.oracle_ce_grad_columns.argtypes = [vp, i64, i64, vp, i64, vp, i64, vp, vp, dbl,
                                                   dbl, vp]
            lib.oracle_ce_grad_columns.restype = None
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = i32
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def count(labels: np.ndarray, V: int, ignore_index: int) -> tuple[int, int]:
    """(n_valid, n_bad): labels in [0, V), and labels neither ignored nor in range."""
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    nv = np.zeros(1, np.int64)
    nb = np.zeros(1, np.int64)
    _load().oracle_ce_count(_ptr(lab), lab.size, V, ignore_index, _ptr(nv), _ptr(nb))
    return int(nv[0]), int(nb[0])


def scale(reduction: str, grad_scale: float, n_valid: int) -> float:
    """Gradient factor of one valid row (mean: grad_scale / n_valid; sum: grad_scale)."""
    return float(_load().oracle_ce_scale(REDUCTIONS[reduction], grad_scale, n_valid))


def rows(x: np.ndarray, dtype: str, V: int, labels: np.ndarray, *, ignore_index: int = -100,
         label_smoothing: float = 0.0, softcap: float = 0.0, row_scale: float = 1.0,
         want_grad: bool = True, threads: int = 0):
    """Per-row (loss fp64 [n], argmax int64 [n], grad fp64 [n, V] or None).

    ``x`` is a 2-D array of stored elements: float32 for "f32", uint16 bit
    patterns (or any 2-byte array) for "bf16", float64 for "f64"; its second
    dimension is the row stride and only the first V columns are read.
    ``row_scale`` multiplies the gradient of every valid row.
    """
    x = np.ascontiguousarray(x)
    assert x.ndim == 2 and x.shape[1] >= V
    assert x.dtype.itemsize == {"f32": 4, "bf16": 2, "f64": 8}[dtype]
    n = x.shape[0]
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    assert lab.shape == (n,)
    loss = np.zeros(n, np.float64)
    amax = np.zeros(n, np.int64)
    grad = np.zeros((n, V), np.float64) if want_grad else None
    rc = _load().oracle_ce_rows(_ptr(x), DTYPES[dtype], n, V, x.shape[1], _ptr(lab), ignore_index,
                                float(label_smoothing), float(softcap), float(row_scale),
                                _ptr(loss), _ptr(amax), _ptr(grad) if want_grad else None,
                                int(threads))
    if rc != 0:
        raise RuntimeError("oracle_ce_rows failed")
    return loss, amax, grad


def reduce(loss: np.ndarray, argmax: np.ndarray, labels: np.ndarray, V: int, ignore_index: int,
           reduction: str) -> tuple[float, float, int]:
    """(reduced loss, accuracy, n_correct), summed in row order in fp64."""
    loss = np.ascontiguousarray(loss, dtype=np.float64)
    amax = np.ascontiguousarray(argmax, dtype=np.int64)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    rl = np.zeros(1, np.float64)
    acc = np.zeros(1, np.float64)
    nc = np.zeros(1, np.int64)
    _load().oracle_ce_reduce(_ptr(loss), _ptr(amax), _ptr(lab), lab.size, V, ignore_index,
                             REDUCTIONS[reduction], _ptr(rl), _ptr(acc), _ptr(nc))
    return float(rl[0]), float(acc[0]), int(nc[0])


def ce_fwd_bwd(x: np.ndarray, dtype: str, V: int, labels: np.ndarray, *, ignore_index: int = -100,
               label_smoothing: float = 0.0, softcap: float = 0.0, reduction: str = "mean",
               grad_scale: float = 1.0, grad_per_token: np.ndarray | None = None,
               want_grad: bool = True, threads: int = 0) -> dict:
    """The whole forward + backward over all rows.

    reduction "mean" / "sum" reduce the per-token losses; "none" keeps them
    (reduced_loss is then their sum) and does not divide the gradient.
    grad_per_token ([n] or None) multiplies each row's gradient: the upstream
    gradient of a "none" reduction, row by row.  Returns a dict with loss [n]
    fp64, argmax [n] int64, grad [n, V] fp64 (or None), reduced_loss, accuracy,
    n_valid, n_correct, n_bad and row_scale (the scale common to all rows).
    """
    n_valid, n_bad = count(labels, V, ignore_index)
    s = scale(reduction, grad_scale, n_valid)
    loss, amax, grad = rows(x, dtype, V, labels, ignore_index=ignore_index,
                            label_smoothing=label_smoothing, softcap=softcap, row_scale=s,
                            want_grad=want_grad, threads=threads)
    if grad is not None and grad_per_token is not None:
        grad *= np.asarray(grad_per_token, np.float64)[:, None]
    red, acc, n_correct = reduce(loss, amax, labels, V, ignore_index, reduction)
    return dict(loss=loss, argmax=amax, grad=grad, reduced_loss=red, accuracy=acc,
                n_valid=n_valid, n_correct=n_correct, n_bad=n_bad, row_scale=s)


def grad_columns(x: np.ndarray, cols: np.ndarray, V: int, labels: np.ndarray, lse: np.ndarray,
                 row_scale: np.ndarray, *, ignore_index: int = -100, label_smoothing: float = 0.0,
                 softcap: float = 0.0) -> np.ndarray:
    """Gradient of columns `cols` (fp64 logits x [n, len(cols)]) given each row's lse and scale."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    n, m = x.shape
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    lab = np.ascontiguousarray(labels, dtype=np.int64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    sc = np.ascontiguousarray(row_scale, dtype=np.float64)
    assert cols.shape == (m,) and lab.shape == (n,) and lse.shape == (n,) and sc.shape == (n,)
    g = np.zeros((n, m), np.float64)
    _load().oracle_ce_grad_columns(_ptr(x), n, m, _ptr(cols), V, _ptr(lab), ignore_index,
                                   _ptr(lse), _ptr(sc), float(label_smoothing), float(softcap),
                                   _ptr(g))
    return g


def round_bf16(values: np.ndarray) -> np.ndarray:
    """fp64 -> bfloat16 bit patterns (uint16), round-to-nearest-even, no double rounding."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.zeros(v.shape, np.uint16)
    _load().oracle_round_bf16(_ptr(v), _ptr(out), v.size)
    return out
