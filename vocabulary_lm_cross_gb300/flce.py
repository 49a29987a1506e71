"""PyTorch-facing binding of flce_fwd_bwd (argument marshalling only).

Every step runs in libvlmce.so's CUDA kernels (the tcgen05 GEMM engine with
the cross-entropy epilogues); this module checks tensors, allocates the
outputs and workspace with PyTorch and calls the C ABI.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import capi

_REDUCTIONS = {"mean": capi.MEAN, "sum": capi.SUM}


@dataclass
class FLCEResult:
    loss: torch.Tensor         # fp32 [N]
    argmax: torch.Tensor       # int64 [N]
    reduced: torch.Tensor      # fp32 [2]: reduced loss, token accuracy
    counts: torch.Tensor       # int64 [4]: n_valid, n_correct, n_bad_labels, device error bits
    grad_hidden: torch.Tensor  # [N, H] in the input dtype: gradient with respect to h' = m h
    grad_weight: torch.Tensor  # fp32 [V, H]


def workspace_bytes(N: int, H: int, V: int, chunk_rows: int | None = None) -> int:
    """Workspace bytes of the vocabulary-chunked schedule, or of the
    row-chunked one when chunk_rows is given."""
    if chunk_rows is None:
        return int(capi.lib().vlmce_flce_workspace_bytes(N, H, V))
    return int(capi.lib().vlmce_flce_rows_workspace_bytes(N, H, V, chunk_rows))


def flce_fwd_bwd(hidden: torch.Tensor, weight: torch.Tensor, labels: torch.Tensor, *,
                 ignore_index: int = -100, label_smoothing: float = 0.0, softcap: float = 0.0,
                 reduction: str = "mean", grad_scale: float = 1.0,
                 grad_weight: torch.Tensor | None = None, accumulate_grad_weight: bool = False,
                 workspace: torch.Tensor | None = None,
                 chunk_rows: int | None = None) -> FLCEResult:
    """Fused linear cross-entropy forward + backward.

    hidden: bf16 CUDA [N, H] (rows may be strided), the hidden states already
        multiplied by the logit multiplier; weight: bf16 CUDA [V, H];
    labels: int64 CUDA [N].  grad_weight (fp32 [V, H], contiguous) is
    allocated unless given; with accumulate_grad_weight it is added to.
    chunk_rows: None for the vocabulary-chunked schedule (flce_fwd_bwd_ex),
        else the rows per block of the row-chunked one (flce_fwd_bwd_rows).
    """
    dtypes = {torch.bfloat16: capi.BF16, torch.float16: capi.F16}
    if hidden.dtype not in dtypes or weight.dtype != hidden.dtype:
        raise TypeError("flce_fwd_bwd takes bf16 or fp16 hidden states and weight of one dtype")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden must be [N, H] and weight [V, H]")
    if labels.dtype != torch.int64 or labels.shape != (hidden.shape[0],):
        raise ValueError("labels must be int64 [N]")
    if hidden.stride(1) != 1 or weight.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    N, H = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    labels = labels.contiguous()
    if grad_weight is None:
        grad_weight = (torch.zeros if accumulate_grad_weight else torch.empty)(
            (V, H), dtype=torch.float32, device=dev)
    if grad_weight.shape != (V, H) or not grad_weight.is_contiguous() or \
            grad_weight.dtype != torch.float32:
        raise ValueError("grad_weight must be a contiguous fp32 [V, H] tensor")
    hs = hidden.stride(0) if N > 1 else H
    grad_hidden = torch.empty_strided((N, H), (hs, 1), dtype=hidden.dtype, device=dev)
    res = FLCEResult(loss=torch.empty(N, dtype=torch.float32, device=dev),
                     argmax=torch.empty(N, dtype=torch.int64, device=dev),
                     reduced=torch.empty(2, dtype=torch.float32, device=dev),
                     counts=torch.empty(4, dtype=torch.int64, device=dev),
                     grad_hidden=grad_hidden, grad_weight=grad_weight)
    if chunk_rows is not None and chunk_rows < 1:
        raise ValueError("chunk_rows must be >= 1")
    need = workspace_bytes(N, H, V, chunk_rows)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
    args = (hidden.data_ptr(), dtypes[hidden.dtype], hs, weight.data_ptr(),
            weight.stride(0) if V > 1 else H,
            labels.data_ptr(), N, H, V, ignore_index, float(label_smoothing), float(softcap),
            _REDUCTIONS[reduction], float(grad_scale), res.loss.data_ptr(), res.argmax.data_ptr(),
            res.reduced.data_ptr(), res.counts.data_ptr(), grad_hidden.data_ptr(),
            grad_weight.data_ptr(), int(accumulate_grad_weight))
    if chunk_rows is None:
        st = capi.lib().flce_fwd_bwd_ex(*args, workspace.data_ptr(), workspace.numel(), stream)
        capi.check(st, "flce_fwd_bwd")
    else:
        st = capi.lib().flce_fwd_bwd_rows(*args, int(chunk_rows), workspace.data_ptr(),
                                          workspace.numel(), stream)
        capi.check(st, "flce_fwd_bwd_rows")
    return res
