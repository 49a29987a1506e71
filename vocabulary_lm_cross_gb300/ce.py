"""PyTorch-facing binding of ce_fwd_bwd (argument marshalling only).

Every step of the computation runs in libvlmce.so's CUDA kernels; this module
only checks tensors, takes their device pointers and the current CUDA stream,
and calls the C ABI.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import capi

_DTYPES = {torch.float32: capi.F32, torch.bfloat16: capi.BF16}
_REDUCTIONS = {"mean": capi.MEAN, "sum": capi.SUM, "none": capi.NONE}


@dataclass
class CEResult:
    """Outputs of one ce_fwd_bwd call (device tensors; the gradient is the logits buffer)."""
    loss: torch.Tensor      # fp32 [N] per-token loss
    argmax: torch.Tensor    # int64 [N]
    reduced: torch.Tensor   # fp32 [2]: reduced loss, token accuracy
    counts: torch.Tensor    # int64 [4]: n_valid, n_correct, n_bad_labels, device error bits


def workspace_bytes(N: int, V: int, dtype: torch.dtype) -> int:
    return int(capi.lib().vlmce_ce_workspace_bytes(N, V, _DTYPES[dtype]))


def describe_plan(N: int, V: int, dtype: torch.dtype, softcap: float = 0.0,
                  aligned_rows: bool = True) -> dict:
    """The launch plan ce_fwd_bwd uses for N rows of V elements on the current device."""
    import ctypes
    out = (ctypes.c_int32 * 6)()
    st = capi.lib().vlmce_ce_describe_plan(N, V, _DTYPES[dtype], float(softcap),
                                           int(aligned_rows), ctypes.cast(out, ctypes.c_void_p))
    capi.check(st, "vlmce_ce_describe_plan")
    keys = ("kernel", "ctas_per_row", "granules_per_cta", "resident", "threads", "smem_bytes")
    d = dict(zip(keys, list(out)))
    d["kernel"] = ("rows", "split")[d["kernel"]]
    return d


def max_vocab(dtype: torch.dtype) -> int:
    return int(capi.lib().vlmce_ce_max_vocab(_DTYPES[dtype]))


def ce_fwd_bwd(logits: torch.Tensor, labels: torch.Tensor, *, ignore_index: int = -100,
               label_smoothing: float = 0.0, softcap: float = 0.0, reduction: str = "mean",
               grad_scale: float = 1.0, grad_per_token: torch.Tensor | None = None,
               compute_grad: bool = True, out: CEResult | None = None,
               workspace: torch.Tensor | None = None) -> CEResult:
    """Fused cross-entropy forward + backward; the gradient overwrites ``logits``.

    logits: CUDA tensor [N, V] (fp32 or bf16) whose rows may be strided
        (``logits.stride(1) == 1``; ``stride(0)`` is the row stride, so a view
        ``buf[:, :V]`` of a padded buffer works).  After the call it holds the
        gradient of ``grad_scale * reduced_loss`` and the input is gone; its
        autograd version counter is bumped so stale uses are caught.
    labels: int64 CUDA tensor [N].
    reduction: "mean", "sum" or "none" (per-token losses; the gradient is not
        averaged and ``reduced[0]`` is the sum of the losses).
    grad_per_token: optional fp32 CUDA tensor [N] multiplying each row's
        gradient (the upstream gradient of a "none" reduction).
    compute_grad: False for a forward-only call (the logits are left unchanged).
    """
    if logits.dim() != 2 or labels.dim() != 1 or labels.shape[0] != logits.shape[0]:
        raise ValueError("logits must be [N, V] and labels [N]")
    if logits.dtype not in _DTYPES:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if labels.dtype != torch.int64:
        raise TypeError("labels must be int64")
    if not logits.is_cuda or not labels.is_cuda or logits.device != labels.device:
        raise ValueError("logits and labels must be CUDA tensors on one device")
    N, V = logits.shape
    if V > 1 and logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")
    row_stride = logits.stride(0) if N > 1 else V
    labels = labels.contiguous()
    dev = logits.device
    if out is None:
        out = CEResult(loss=torch.empty(N, dtype=torch.float32, device=dev),
                       argmax=torch.empty(N, dtype=torch.int64, device=dev),
                       reduced=torch.empty(2, dtype=torch.float32, device=dev),
                       counts=torch.empty(4, dtype=torch.int64, device=dev))
    need = workspace_bytes(N, V, logits.dtype)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    gpt = None
    if grad_per_token is not None:
        if grad_per_token.shape != (N,) or grad_per_token.dtype != torch.float32 or \
                not grad_per_token.is_contiguous() or grad_per_token.device != dev:
            raise ValueError("grad_per_token must be a contiguous fp32 [N] tensor on the device")
        gpt = grad_per_token.data_ptr()
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
    st = capi.lib().ce_fwd_bwd_ex(
        logits.data_ptr(), _DTYPES[logits.dtype], labels.data_ptr(), N, V, row_stride,
        ignore_index, float(label_smoothing), float(softcap), _REDUCTIONS[reduction],
        float(grad_scale), gpt, int(bool(compute_grad)), out.loss.data_ptr(),
        out.argmax.data_ptr(), out.reduced.data_ptr(), out.counts.data_ptr(),
        workspace.data_ptr(), workspace.numel(), stream)
    capi.check(st, "ce_fwd_bwd")
    if compute_grad:
        try:
            torch.autograd.graph.increment_version(logits)
        except Exception:  # older/newer torch without the helper: nothing to bump
            pass
    return out


def host_workspace_bytes(N: int, V: int, row_stride: int, dtype: torch.dtype) -> int:
    """Device workspace of ce_fwd_bwd_host with host logits (includes its staging ring)."""
    return int(capi.lib().vlmce_ce_host_workspace_bytes(N, V, row_stride, _DTYPES[dtype]))


def ce_fwd_bwd_host(logits: torch.Tensor, labels: torch.Tensor, *, device: torch.device | str = "cuda",
                    ignore_index: int = -100, label_smoothing: float = 0.0, softcap: float = 0.0,
                    reduction: str = "mean", grad_scale: float = 1.0, out: CEResult | None = None,
                    workspace: torch.Tensor | None = None) -> CEResult:
    """``ce_fwd_bwd`` on page-locked host tensors: the logits stream through
    ``device`` in chunks of rows (copy in, row kernel, gradient copied back
    into ``logits``), labels and outputs are read and written in place.

    logits: pinned CPU tensor [N, V] (fp32 or bf16, rows may be strided);
    labels: pinned int64 CPU tensor [N]; ``out`` tensors (allocated pinned on
    the host unless given) and the gradient in ``logits`` are valid once the
    device's current stream has been synchronised.
    """
    if logits.dim() != 2 or labels.dim() != 1 or labels.shape[0] != logits.shape[0]:
        raise ValueError("logits must be [N, V] and labels [N]")
    if logits.dtype not in _DTYPES:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if labels.dtype != torch.int64:
        raise TypeError("labels must be int64")
    if logits.is_cuda or labels.is_cuda or not logits.is_pinned() or not labels.is_pinned():
        raise ValueError("logits and labels must be page-locked (pinned) CPU tensors")
    N, V = logits.shape
    if V > 1 and logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")
    if not labels.is_contiguous():
        raise ValueError("labels must be contiguous")
    row_stride = logits.stride(0) if N > 1 else V
    dev = torch.device(device)
    if out is None:
        out = CEResult(loss=torch.empty(N, dtype=torch.float32).pin_memory(),
                       argmax=torch.empty(N, dtype=torch.int64).pin_memory(),
                       reduced=torch.empty(2, dtype=torch.float32).pin_memory(),
                       counts=torch.empty(4, dtype=torch.int64).pin_memory())
    need = host_workspace_bytes(N, V, row_stride, logits.dtype)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = capi.lib().ce_fwd_bwd_host(
            logits.data_ptr(), _DTYPES[logits.dtype], labels.data_ptr(), N, V, row_stride,
            ignore_index, float(label_smoothing), float(softcap), _REDUCTIONS[reduction],
            float(grad_scale), out.loss.data_ptr(), out.argmax.data_ptr(), out.reduced.data_ptr(),
            out.counts.data_ptr(), workspace.data_ptr(), workspace.numel(), stream)
    capi.check(st, "ce_fwd_bwd_host")
    return out
