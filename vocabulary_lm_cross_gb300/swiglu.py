"""PyTorch-facing binding of the fused gate-up SwiGLU (argument marshalling
only): swiglu_fwd / swiglu_bwd of libvlmce.so on the [tokens, 2n] layout
(gate | up) of a fused first linear layer."""
from __future__ import annotations

import torch

from . import capi
from .ce import _DTYPES


def _stream(dev):
    with torch.cuda.device(dev):
        return torch.cuda.current_stream(dev).cuda_stream


def _rows(t: torch.Tensor, name: str):
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be [T, columns] with contiguous rows")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def swiglu_fwd(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """y [T, n] = silu(x[:, :n]) * x[:, n:2n] for x [T, 2n] (bf16 or fp32, CUDA)."""
    if x.dtype not in _DTYPES or not x.is_cuda:
        raise TypeError("x must be a bf16 or fp32 CUDA tensor")
    T, c = x.shape
    if c % 2:
        raise ValueError("x must have 2n columns")
    n = c // 2
    xs = _rows(x, "x")
    if out is None:
        out = torch.empty((T, n), dtype=x.dtype, device=x.device)
    ys = _rows(out, "out")
    st = capi.lib().swiglu_fwd(x.data_ptr(), _DTYPES[x.dtype], T, n, xs, out.data_ptr(), ys,
                               _stream(x.device))
    capi.check(st, "swiglu_fwd")
    return out


def swiglu_bwd(x: torch.Tensor, dy: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """dx [T, 2n] = (d_gate | d_up) for dy [T, n]; ``out=x`` works in place."""
    if x.dtype not in _DTYPES or dy.dtype != x.dtype or not x.is_cuda or not dy.is_cuda:
        raise TypeError("x and dy must be CUDA tensors of one dtype (bf16 or fp32)")
    T, c = x.shape
    n = c // 2
    if c % 2 or dy.shape != (T, n):
        raise ValueError("x must be [T, 2n] and dy [T, n]")
    xs, ds = _rows(x, "x"), _rows(dy, "dy")
    if out is None:
        out = torch.empty((T, 2 * n), dtype=x.dtype, device=x.device)
    os_ = _rows(out, "out")
    st = capi.lib().swiglu_bwd(x.data_ptr(), xs, dy.data_ptr(), ds, out.data_ptr(), os_,
                               _DTYPES[x.dtype], T, n, _stream(x.device))
    capi.check(st, "swiglu_bwd")
    return out
