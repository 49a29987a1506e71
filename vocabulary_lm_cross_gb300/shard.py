"""PyTorch-facing binding of the vocabulary-sharded cross-entropy (argument
marshalling only): ce_shard_stats, ce_merge_stats and ce_shard_fwd_bwd of
libvlmce.so.  Row statistics travel as float32 tensors [N, 8] (32 bytes a
row, the layout of vlmce_row_stats: x_max, argmax as int32 bits, m, s, sum_z,
z_y, two reserved words), so they can be all-gathered like any tensor.
"""
from __future__ import annotations

import torch

from . import capi
from .ce import _DTYPES, _REDUCTIONS, CEResult, workspace_bytes


def _stream(dev):
    with torch.cuda.device(dev):
        return torch.cuda.current_stream(dev).cuda_stream


def _check(logits, labels):
    if logits.dim() != 2 or labels.dim() != 1 or labels.shape[0] != logits.shape[0]:
        raise ValueError("logits must be [N, V_local] and labels [N]")
    if logits.dtype not in _DTYPES:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if labels.dtype != torch.int64 or not labels.is_contiguous():
        raise ValueError("labels must be a contiguous int64 tensor")
    if not logits.is_cuda or not labels.is_cuda:
        raise ValueError("logits and labels must be CUDA tensors")
    if logits.shape[1] > 1 and logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")


def _stats_out(out, N, dev):
    if out is None:
        return torch.empty((N, 8), dtype=torch.float32, device=dev)
    if out.shape != (N, 8) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 [N, 8] tensor")
    return out


def shard_stats(logits: torch.Tensor, labels: torch.Tensor, vocab_start: int, V: int, *,
                softcap: float = 0.0, out: torch.Tensor | None = None) -> torch.Tensor:
    """Row statistics [N, 8] of the shard (columns vocab_start.. of the vocabulary V),
    written to ``out`` if given (e.g. this rank's slot of an all-gather buffer)."""
    _check(logits, labels)
    N, VL = logits.shape
    out = _stats_out(out, N, logits.device)
    st = capi.lib().ce_shard_stats(logits.data_ptr(), _DTYPES[logits.dtype], labels.data_ptr(), N,
                                   VL, logits.stride(0) if N > 1 else VL, vocab_start, V,
                                   float(softcap), out.data_ptr(), _stream(logits.device))
    capi.check(st, "ce_shard_stats")
    return out


def merge_stats(shards: torch.Tensor, *, out: torch.Tensor | None = None) -> torch.Tensor:
    """Merge [k, N, 8] statistics in shard order into [N, 8] (``out`` if given)."""
    if shards.dim() != 3 or shards.shape[2] != 8 or shards.dtype != torch.float32:
        raise ValueError("shards must be float32 [k, N, 8]")
    if not shards.is_contiguous():
        raise ValueError("shards must be contiguous")
    k, N, _ = shards.shape
    out = _stats_out(out, N, shards.device)
    st = capi.lib().ce_merge_stats(shards.data_ptr(), k, N, out.data_ptr(), _stream(shards.device))
    capi.check(st, "ce_merge_stats")
    return out


def shard_fwd_bwd(logits: torch.Tensor, labels: torch.Tensor, vocab_start: int, V: int,
                  stats: torch.Tensor, *, ignore_index: int = -100,
                  label_smoothing: float = 0.0, softcap: float = 0.0, reduction: str = "mean",
                  grad_scale: float = 1.0, out: CEResult | None = None,
                  workspace: torch.Tensor | None = None) -> CEResult:
    """Loss and the shard's gradient (written over ``logits``) from the whole
    vocabulary's statistics: ``stats`` is either the merged [N, 8] records
    (ce_shard_fwd_bwd) or the gathered [k, N, 8] records of every shard in
    shard order, merged inside the gradient kernel (ce_shard_fwd_bwd_gathered)."""
    _check(logits, labels)
    N, VL = logits.shape
    dev = logits.device
    gathered = stats.dim() == 3
    ok_shape = (stats.shape[1:] == (N, 8)) if gathered else (stats.shape == (N, 8))
    if not ok_shape or stats.dtype != torch.float32 or not stats.is_contiguous():
        raise ValueError("stats must be a contiguous float32 [N, 8] or [k, N, 8] tensor")
    if out is None:
        out = CEResult(loss=torch.empty(N, dtype=torch.float32, device=dev),
                       argmax=torch.empty(N, dtype=torch.int64, device=dev),
                       reduced=torch.empty(2, dtype=torch.float32, device=dev),
                       counts=torch.empty(4, dtype=torch.int64, device=dev))
    need = workspace_bytes(N, V, logits.dtype)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    head = (logits.data_ptr(), _DTYPES[logits.dtype], labels.data_ptr(), N, VL,
            logits.stride(0) if N > 1 else VL, vocab_start, V, ignore_index,
            float(label_smoothing), float(softcap), _REDUCTIONS[reduction], float(grad_scale))
    tail = (out.loss.data_ptr(), out.argmax.data_ptr(), out.reduced.data_ptr(),
            out.counts.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(dev))
    if gathered:
        st = capi.lib().ce_shard_fwd_bwd_gathered(*head, stats.data_ptr(), stats.shape[0], *tail)
    else:
        st = capi.lib().ce_shard_fwd_bwd(*head, stats.data_ptr(), *tail)
    capi.check(st, "shard_fwd_bwd")
    try:
        torch.autograd.graph.increment_version(logits)
    except Exception:
        pass
    return out
