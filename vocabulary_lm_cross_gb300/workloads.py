"""Seeded synthetic workloads for the fused LM cross-entropy.

This module only draws inputs; it holds none of the method's arithmetic, so
both the CUDA path's tests and the oracle may use it.  Every array is drawn
from a seeded ``torch.Generator`` on the requested device: fp32 normal
samples, rounded to the storage dtype with round-to-nearest-even by
``Tensor.to``.  The shapes and value distributions stand in for the training
batches the pages measure on (Qwen3 vocabulary 151,936 at sequence 4096 x
micro-batch 2; sequence 2048 with a 128K vocabulary; Muse Glimmer's hidden
size 6656 and vocabulary 202,048); no dataset or trained weight is used.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

IGNORE_INDEX = -100

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class CEWorkload:
    """One cross-entropy workload: logits [N, V] in rows of ``row_stride`` elements."""
    name: str
    N: int
    V: int
    dtype: str                 # "f32" | "bf16"
    sigma: float               # logits ~ N(0, sigma^2)
    ignore_frac: float         # exactly round(ignore_frac * N) rows get ignore_index
    label_smoothing: float
    softcap: float             # 0 = off
    reduction: str             # "mean" | "sum"
    grad_scale: float
    seed: int
    row_stride: int = 0        # 0 = V (contiguous rows)
    label_boost: float = 0.0   # added (in fp32, before rounding) to the label logit of half the rows
    dup_max_frac: float = 0.0  # fraction of rows given an exact duplicate of their maximum
    want_argmax: bool = False
    pad_value: float = float("nan")  # value of the padding columns [V, row_stride)

    @property
    def stride(self) -> int:
        return self.row_stride or self.V

    @property
    def elt_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def algorithmic_bytes(self) -> int:
        """One read plus one write of the N x V logits (padding excluded)."""
        return 2 * self.N * self.V * self.elt_bytes

    def resized(self, N: int | None = None, V: int | None = None, row_stride: int | None = None,
                seed: int | None = None) -> "CEWorkload":
        kw = {}
        if N is not None:
            kw["N"] = N
        if V is not None:
            kw["V"] = V
            kw["row_stride"] = 0
        if row_stride is not None:
            kw["row_stride"] = row_stride
        if seed is not None:
            kw["seed"] = seed
        return replace(self, **kw)


@dataclass(frozen=True)
class FLCEWorkload:
    """Fused linear cross-entropy: hidden [N, H] (pre-scaled by m), weight [V, H]."""
    name: str
    N: int
    H: int
    V: int
    hidden_sigma: float
    weight_sigma: float
    multiplier: float          # m, folded into the hidden states (exact in bf16 for 0.5)
    ignore_frac: float
    label_smoothing: float
    softcap: float
    reduction: str
    grad_scale: float
    seed: int
    dtype: str = "bf16"        # "bf16" | "f16": hidden states, weight, grad_hidden

    @property
    def algorithmic_flops(self) -> int:
        """6 N V H: the logits GEMM and the two gradient GEMMs."""
        return 6 * self.N * self.V * self.H

    def resized(self, N=None, H=None, V=None, seed=None, dtype=None) -> "FLCEWorkload":
        kw = {k: v for k, v in dict(N=N, H=H, V=V, seed=seed, dtype=dtype).items() if v is not None}
        return replace(self, **kw)


CE_WORKLOADS = {
    w.name: w for w in [
        CEWorkload("ce-f32-256x4096", N=256, V=4096, dtype="f32", sigma=1.0, ignore_frac=0.05,
                   label_smoothing=0.0, softcap=0.0, reduction="mean", grad_scale=1.0, seed=1001),
        CEWorkload("ce-bf16-8192x32000", N=8192, V=32000, dtype="bf16", sigma=2.0,
                   ignore_frac=0.10, label_smoothing=0.0, softcap=0.0, reduction="mean",
                   grad_scale=1.0, seed=1002),
        CEWorkload("ce-bf16-2048x131072-ls0.1-argmax", N=2048, V=131072, dtype="bf16", sigma=3.0,
                   ignore_frac=0.03, label_smoothing=0.1, softcap=0.0, reduction="mean",
                   grad_scale=1.0, seed=1003, label_boost=4.0, dup_max_frac=0.01,
                   want_argmax=True),
        CEWorkload("ce-bf16-8192x151936-stride152064-softcap30-sum", N=8192, V=151936,
                   dtype="bf16", sigma=4.0, ignore_frac=0.05, label_smoothing=0.1, softcap=30.0,
                   reduction="sum", grad_scale=1.0 / 4096, seed=1004, row_stride=152064),
        # few wide rows (the V-split kernel's case: a cluster of CTAs per row),
        # e.g. an evaluation batch of 32 tokens over the Qwen3 vocabulary
        CEWorkload("ce-bf16-32x151936-ls0.1-argmax", N=32, V=151936, dtype="bf16", sigma=3.0,
                   ignore_frac=0.05, label_smoothing=0.1, softcap=0.0, reduction="mean",
                   grad_scale=1.0, seed=1009, label_boost=4.0, dup_max_frac=0.1,
                   want_argmax=True),
        # the headline recipe at a profiling size (268 MB, still larger than L2)
        CEWorkload("ce-bf16-1024x131072-ls0.1-argmax", N=1024, V=131072, dtype="bf16", sigma=3.0,
                   ignore_frac=0.03, label_smoothing=0.1, softcap=0.0, reduction="mean",
                   grad_scale=1.0, seed=1008, label_boost=4.0, dup_max_frac=0.01,
                   want_argmax=True),
        # the same recipe at a profiling size (311 MB, still larger than L2)
        CEWorkload("ce-bf16-1024x151936-stride152064-softcap30-sum", N=1024, V=151936,
                   dtype="bf16", sigma=4.0, ignore_frac=0.05, label_smoothing=0.1, softcap=30.0,
                   reduction="sum", grad_scale=1.0 / 4096, seed=1007, row_stride=152064),
    ]
}

# The workload the headline metric is quoted on: N = 2048 (sequence 2048 x batch 1), V = 131072.
HEADLINE_CE = "ce-bf16-2048x131072-ls0.1-argmax"

FLCE_WORKLOADS = {
    w.name: w for w in [
        FLCEWorkload("flce-bf16-4096x6656x202048-softcap30", N=4096, H=6656, V=202048,
                     hidden_sigma=1.0, weight_sigma=0.02, multiplier=0.5, ignore_frac=0.02,
                     label_smoothing=0.0, softcap=30.0, reduction="mean", grad_scale=1.0,
                     seed=1005),
        # the same recipe at a profiling size (weight 436 MB, still larger than L2)
        FLCEWorkload("flce-bf16-1024x6656x32768-softcap30", N=1024, H=6656, V=32768,
                     hidden_sigma=1.0, weight_sigma=0.02, multiplier=0.5, ignore_frac=0.02,
                     label_smoothing=0.0, softcap=30.0, reduction="mean", grad_scale=1.0,
                     seed=1006),
    ]
}


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def make_ce_inputs(w: CEWorkload, device="cpu"):
    """(logits, labels): logits [N, row_stride] in w.dtype, labels int64 [N].

    Recipe: x ~ N(0, sigma^2) in fp32; labels uniform in [0, V); on a random
    half of the rows the label logit gets +label_boost (fp32, before
    rounding); x is rounded to the storage dtype (RNE); on round(dup_max_frac
    N) rows the row maximum is copied to a second column, alternately to the
    left and to the right of the first maximum, and half of those rows are
    rows whose maximum sits on the label when there are such rows; exactly
    round(ignore_frac N) rows (a random permutation) get ignore_index;
    padding columns [V, row_stride) hold pad_value.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    cg = _cpu_gen(w.seed + 7919)
    N, V, S = w.N, w.V, w.stride
    x = torch.randn((N, V), generator=g, device=dev, dtype=torch.float32)
    x.mul_(w.sigma)
    labels = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int64)
    if w.label_boost and N > 0:
        rows = torch.randperm(N, generator=cg)[: N // 2].to(dev)
        x[rows, labels[rows]] += w.label_boost
    store = torch.full((N, S), w.pad_value, dtype=_TORCH_DTYPE[w.dtype], device=dev)
    store[:, :V] = x.to(_TORCH_DTYPE[w.dtype])
    del x
    n_dup = int(round(w.dup_max_frac * N))
    if n_dup and V >= 2:
        amax = store[:, :V].float().argmax(dim=1)
        on_label = torch.nonzero(amax == labels).flatten().cpu()
        others = torch.nonzero(amax != labels).flatten().cpu()
        on_label = on_label[torch.randperm(on_label.numel(), generator=cg)]
        others = others[torch.randperm(others.numel(), generator=cg)]
        take = min(n_dup // 2, on_label.numel())
        chosen = torch.cat([on_label[:take], others[: n_dup - take]]).tolist()
        amax_h = amax.cpu()
        for i, r in enumerate(chosen):
            a = int(amax_h[r])
            left = (i % 2 == 0 and a > 0) or a == V - 1
            if left:
                col = int(torch.randint(0, a, (1,), generator=cg))
            else:
                col = int(torch.randint(a + 1, V, (1,), generator=cg))
            store[r, col] = store[r, a]
    n_ign = int(round(w.ignore_frac * N))
    if n_ign:
        ign = torch.randperm(N, generator=cg)[:n_ign].to(dev)
        labels[ign] = IGNORE_INDEX
    return store, labels


def make_flce_inputs(w: FLCEWorkload, device="cpu"):
    """(hidden, weight, labels): hidden [N, H] in w.dtype (bf16 or fp16),
    already multiplied by m (exact for m = 0.5), weight [V, H] in w.dtype,
    labels int64 [N] with exactly round(ignore_frac N) ignored rows."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    cg = _cpu_gen(w.seed + 7919)
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    h = torch.randn((w.N, w.H), generator=g, device=dev, dtype=torch.float32)
    h.mul_(w.hidden_sigma)
    hb = h.to(dt)
    del h
    hb.mul_(w.multiplier)
    W = torch.empty((w.V, w.H), device=dev, dtype=dt)
    chunk = max(1, (1 << 28) // max(1, w.H))
    for v0 in range(0, w.V, chunk):
        v1 = min(w.V, v0 + chunk)
        t = torch.randn((v1 - v0, w.H), generator=g, device=dev, dtype=torch.float32)
        W[v0:v1] = (t * w.weight_sigma).to(dt)
    labels = torch.randint(0, w.V, (w.N,), generator=g, device=dev, dtype=torch.int64)
    n_ign = int(round(w.ignore_frac * w.N))
    if n_ign:
        ign = torch.randperm(w.N, generator=cg)[:n_ign].to(dev)
        labels[ign] = IGNORE_INDEX
    return hb, W, labels


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's storage as a numpy uint16 array (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
